"""pkv_paged_decode_attention_static: the allocation-free variant of the batched
entry point, for callers that cannot allocate device memory (an application
that already reserved the GPU's memory for its own arena, or a latency-critical
path that must not call cudaMalloc).  Its scratch is a fixed device array inside
the library.  Checked through the C ABI against pkv_paged_decode_attention, on
calls in a row that reuse the array with the previous call's contents in it.
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


@pytest.mark.parametrize("lens,H,D,dtype", [
    ([1, 17, 300, 4096, 64, 1000, 33, 2048], 8, 128, BF16),
    ([5, 16, 129, 700], 4, 64, F32),
])
def test_static_scratch_matches_workspace_entry(lens, H, D, dtype):
    run = BatchedRun(make_workload("static", lens, H, D, dtype=dtype, seed=31))
    try:
        ref = run.run().clone()
        assert run.pool.check_device_status() == 0
        for _ in range(2):                         # two calls in a row share the array
            out = torch.full_like(ref, float("nan"))
            assert call_static(run, out) == pkv.PKV_OK, pkv.lib.pkv_last_error()
            torch.cuda.synchronize()
            assert run.pool.check_device_status() == 0
            check_close(out.cpu().numpy(), ref.cpu().numpy().astype(np.float64), dtype, "static")
    finally:
        run.close()


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
