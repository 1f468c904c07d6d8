"""Replica ranks of bench.py: timing max over ranks and barriers, world size 2 on
CPU with the gloo backend (no GPU, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, w = bench.dist_init("gloo")
    bench.barrier()
    mx = bench.max_over_ranks(1.5 + rank)
    # each replica draws its own inputs
    wl = bench.make_workload("batched_bf16", r)
    q.put((r, w, mx, wl.seed))
    bench.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got)
    assert all(g[2] == 2.5 for g in got)            # max over ranks
    assert got[0][3] != got[1][3]                   # distinct replica seeds


def test_single_process_helpers_are_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    bench.barrier()
    assert bench.dist_env()[1] >= 1
