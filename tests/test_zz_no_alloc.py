"""pkv_paged_decode_attention_static: the allocation-free variant of the batched
entry point, for callers that cannot allocate device memory (an application
that already reserved the GPU's memory for its own arena, or a latency-critical
path that must not call cudaMalloc).  Its scratch is a fixed device array inside
the library.  Checked through the C ABI against the oracle and against
pkv_paged_decode_attention, on calls in a row that reuse the array with an
earlier call's contents in it.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_decode_gb300 as pkv
from synth import F32, BF16
from tests._gpu import BatchedRun, check_close, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def call_static(run, out):
    d = run.dev
    return pkv.lib.pkv_paged_decode_attention_static(
        run.pool.handle, 0, run.w.B, _p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["tables"]),
        d["tables"].shape[1], _p(d["lens"]), run.max_seq_len, _p(out),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def oracle_array(run):
    """The oracle's output of every (request, query head) row: [B, HQ, D] fp64."""
    ref = run.oracle_out()
    w = run.w
    return np.stack([np.stack([ref[(b, h)] for h in range(w.HQ)]) for b in range(w.B)])


def static_twice_checked(run, dtype, what):
    """Two static calls in a row, each checked against the oracle and against the
    workspace entry point's output of the same step."""
    ref = run.run().clone()
    assert run.pool.check_device_status() == 0
    orc = oracle_array(run)
    check_close(ref.cpu().numpy(), orc, dtype, what + " workspace entry vs oracle")
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        assert call_static(run, out) == pkv.PKV_OK, pkv.lib.pkv_last_error()
        torch.cuda.synchronize()
        assert run.pool.check_device_status() == 0
        got = out.cpu().numpy()
        check_close(got, orc, dtype, f"{what} static call {call} vs oracle")
        check_close(got, ref.cpu().numpy().astype(np.float64), dtype,
                    f"{what} static call {call} vs workspace entry")


@pytest.mark.parametrize("lens,H,D,dtype,group", [
    ([1, 17, 300, 4096, 64, 1000, 33, 2048], 8, 128, BF16, 1),
    ([5, 16, 129, 700], 4, 64, F32, 1),
    ([3, 250, 1500, 4000, 16, 17], 2, 128, BF16, 8),     # tensor-core kernel, lanes of 8 rows
])
def test_static_scratch_matches_workspace_entry(lens, H, D, dtype, group):
    run = BatchedRun(make_workload("static", lens, H, D, dtype=dtype, seed=31, group=group))
    try:
        static_twice_checked(run, dtype, f"G={group}")
    finally:
        run.close()


def test_static_scratch_after_a_larger_call():
    """A long many-lane call fills much of the array with partials; a smaller call
    of another shape must then read none of them (its own merge only)."""
    big = BatchedRun(make_workload("big", [8192, 6000, 8191, 7777] * 4, 8, 128, dtype=BF16,
                                   seed=33))
    try:
        out = torch.full_like(big.out, float("nan"))
        assert call_static(big, out) == pkv.PKV_OK, pkv.lib.pkv_last_error()
        torch.cuda.synchronize()
        assert big.pool.check_device_status() == 0
        assert torch.isfinite(out).all()
    finally:
        big.close()
    small = BatchedRun(make_workload("small", [40, 900, 2], 4, 64, dtype=F32, seed=34, group=2))
    try:
        static_twice_checked(small, F32, "after a larger call")
    finally:
        small.close()


def test_static_scratch_rejects_batches_beyond_its_size():
    run = BatchedRun(make_workload("small", [20, 40], 32, 128, dtype=BF16, seed=32))
    try:
        huge_batch = 4096                          # 4096 x 32 lanes of partials > 8 MiB
        need = run.pool.workspace_size(huge_batch, 1 << 17)
        assert need > (8 << 20)
        out = torch.full((2, 32, 128), float("nan"), device="cuda")
        d = run.dev
        st = pkv.lib.pkv_paged_decode_attention_static(
            run.pool.handle, 0, huge_batch, _p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["tables"]),
            d["tables"].shape[1], _p(d["lens"]), 1 << 17, _p(out), None)
        assert st == pkv.PKV_ERR_INVALID_ARGUMENT
        assert b"static array" in pkv.lib.pkv_last_error()
        torch.cuda.synchronize()
        assert torch.isnan(out).all()
        assert run.pool.check_device_status() == 0
    finally:
        run.close()
