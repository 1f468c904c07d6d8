"""Shared-prefix decode (prefix pass on the tensor cores + the split kernel over each
request's own positions, merged) vs the fp64 oracle, through the C ABI.

Bar: the same as the batched decode path — bit-exact appended rows; bf16 storage
normwise relative error per (request, query head) row <= 5e-3 — and, since the
prefix pass splits q and the weights into bf16 hi + lo, agreement with the plain
batched call to 1e-4.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_decode_gb300 as pkv
from synth import BF16, F32, workloads
from synth.workloads import Workload
from tests._gpu import BatchedRun, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _workload(name, B, prefix, suffix_max, H, D, G, window=0, seed=0, P=16):
    rng = np.random.default_rng(seed)
    lens = (prefix + rng.integers(1, suffix_max + 1, size=B)).astype(np.int32)
    pages = int(((lens.astype(np.int64) + P - 1) // P).sum()) + 16
    return Workload(name, B, 1, H, D, P, BF16, pages, int(lens.max()), seed, lens, group=G,
                    window=window, shared_prefix=prefix)


def _shared(run, prefix):
    d = run.dev
    return run.pool.paged_decode_attention_shared(0, d["q"], d["k"], d["v"], d["tables"], d["lens"],
                                                  run.max_seq_len, prefix)


CASES = {
    # name: (B, prefix, suffix_max, H, D, G, window)
    "g4_d128": (6, 256, 100, 2, 128, 4, 0),
    "g1_d64": (5, 320, 40, 2, 64, 1, 0),
    "g8_d128_many_rows": (40, 144, 300, 1, 128, 8, 0),
    "g2_d64_window": (7, 512, 90, 2, 64, 2, 200),
    "g4_d128_short_prefix": (3, 16, 17, 2, 128, 4, 0),
    "g16_d128_mqa": (9, 192, 60, 2, 128, 16, 0),
    "g32_d64_mqa_window": (5, 128, 70, 1, 64, 32, 90),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_shared_prefix_matches_oracle(name):
    B, prefix, smax, H, D, G, W = CASES[name]
    w = _workload(name, B, prefix, smax, H, D, G, W, seed=len(name))
    run = BatchedRun(w)
    try:
        out = _shared(run, prefix).cpu().numpy()
        torch.cuda.synchronize()
        assert run.pool.check_device_status() == 0
        ref = run.oracle_out()
        err = check_close(np.stack([out[k] for k in ref]), np.stack(list(ref.values())), BF16, name)
        for b in range(B):
            k, v = run.appended_rows(b)
            assert k.tobytes() == run.k_new[b].tobytes() and v.tobytes() == run.v_new[b].tobytes()
        plain = run.run().cpu().numpy()
        num = np.abs(out - plain).max(axis=-1)
        den = np.maximum(np.abs(plain).max(axis=-1), 1e-6)
        agree = float((num / den).max())
        print(f"{name}: oracle error {err:.2e}, vs plain call {agree:.2e}")
        assert agree <= 1e-4
    finally:
        run.close()


def test_shared_prefix_table_mismatch_sets_error_bit():
    w = _workload("mismatch", 4, 64, 20, 2, 128, 4, seed=3)
    run = BatchedRun(w)
    try:
        tables = run.dev["tables"].clone()
        tables[2, 1] = tables[2, 4]            # request 2 points one prefix page elsewhere
        d = run.dev
        run.pool.paged_decode_attention_shared(0, d["q"], d["k"], d["v"], tables, d["lens"],
                                               run.max_seq_len, 64)
        torch.cuda.synchronize()
        with pytest.raises(pkv.PkvError) as e:
            run.pool.check_device_status()
        assert "0x8" in str(e.value)
    finally:
        run.close()


def test_shared_prefix_full_workload_sampled():
    """The 64-request shared-prompt workload at full size: sampled requests against the
    oracle, every output finite."""
    w = workloads.shared_prompt()
    run = BatchedRun(w)
    try:
        out = _shared(run, w.shared_prefix)
        torch.cuda.synchronize()
        assert run.pool.check_device_status() == 0
        assert torch.isfinite(out).all()
        out = out.cpu().numpy()
        reqs = [0, 1, 31, 63]
        ref = run.oracle_out(requests=reqs)
        err = check_close(np.stack([out[k] for k in ref]), np.stack(list(ref.values())), BF16,
                          "prefix_bf16 shared")
        print(f"prefix_bf16 shared sampled: {err:.2e}")
    finally:
        run.close()


def test_shared_prefix_edge_lengths_and_page_size():
    """A request whose only own position is its new token, page size 32, a window that
    cuts into the prefix for some requests, G = 1 (CUDA-core suffix kernel)."""
    rng_lens = [1, 2, 40, 97]                       # own positions (the new token included)
    prefix = 96
    lens = np.array([prefix + n for n in rng_lens], dtype=np.int32)
    pages = int(((lens.astype(np.int64) + 31) // 32).sum()) + 8
    w = Workload("edge", len(lens), 1, 2, 64, 32, BF16, pages, int(lens.max()), 17, lens, group=1,
                 window=60, shared_prefix=prefix)
    run = BatchedRun(w)
    try:
        out = _shared(run, prefix).cpu().numpy()
        torch.cuda.synchronize()
        assert run.pool.check_device_status() == 0
        ref = run.oracle_out()
        check_close(np.stack([out[k] for k in ref]), np.stack(list(ref.values())), BF16, "edge")
    finally:
        run.close()


def test_shared_prefix_request_without_own_positions_sets_error_bit():
    w = _workload("short", 3, 64, 10, 2, 128, 4, seed=8)
    run = BatchedRun(w)
    try:
        lens = run.dev["lens"].clone()
        lens[1] = 64                                    # t_b == shared_len: its new row would be shared
        d = run.dev
        run.pool.paged_decode_attention_shared(0, d["q"], d["k"], d["v"], d["tables"], lens,
                                               run.max_seq_len, 64)
        torch.cuda.synchronize()
        with pytest.raises(pkv.PkvError) as e:
            run.pool.check_device_status()
        assert "0x1" in str(e.value)
    finally:
        run.close()


def test_shared_prefix_argument_errors():
    w = _workload("args", 2, 32, 5, 2, 128, 4, seed=9)
    run = BatchedRun(w)
    try:
        d = run.dev
        for shared, st in [(17, pkv.PKV_ERR_INVALID_ARGUMENT), (run.max_seq_len, pkv.PKV_ERR_INVALID_ARGUMENT)]:
            with pytest.raises(pkv.PkvError) as e:
                run.pool.paged_decode_attention_shared(0, d["q"], d["k"], d["v"], d["tables"], d["lens"],
                                                       run.max_seq_len, shared)
            assert e.value.status == st
    finally:
        run.close()
    # fp32 pools have no shared-prefix kernel: the call is the plain batched one
    w32 = Workload("f32", 2, 1, 2, 64, 16, 0, 64, 256, 1, np.array([40, 50], dtype=np.int32),
                   shared_prefix=32)
    run = BatchedRun(w32)
    try:
        d = run.dev
        out = run.pool.paged_decode_attention_shared(0, d["q"], d["k"], d["v"], d["tables"],
                                                     d["lens"], run.max_seq_len, 32)
        torch.cuda.synchronize()
        assert run.pool.check_device_status() == 0
        ref = run.oracle_out()
        check_close(np.stack([out.cpu().numpy()[k] for k in ref]), np.stack(list(ref.values())),
                    F32, "fp32 shared call")
    finally:
        run.close()
