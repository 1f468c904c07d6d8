"""CUDA path vs the fp64 oracle, through the C ABI, on the same seeded inputs.

Bar: bit-exact page tables, visible lengths and appended K/V bytes; max abs
error <= 1e-5 for fp32 storage; normwise relative error per (request, head)
row <= 5e-3 for bf16 storage (fp32 accumulation on the device).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_decode_gb300 as pkv
import synth
from oracle.model import OraclePool
from synth import F32, BF16, KHIST, VHIST, Q, workloads
from synth.device import to_device
from tests._gpu import BatchedRun, check_close, make_workload, dtype_name, FP32_ATOL

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _host(t: torch.Tensor, dtype: int) -> np.ndarray:
    t = t.cpu()
    if dtype == BF16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


# ------------------------------------------------------------ transactional --

def _lane_tensors(seed, layer, H, pos, D, dtype, kseed=None, group=1):
    kseed = seed if kseed is None else kseed
    q = synth.lane_rows(seed, Q, layer, 0, H * group, pos, D, F32)
    k = synth.lane_rows(kseed, KHIST, layer, 0, H, pos, D, dtype)
    v = synth.lane_rows(kseed, VHIST, layer, 0, H, pos, D, dtype)
    return q, k, v


def _serial(layers, H, D, dtype, pool_pages, max_context, steps, seed, abort_at=None,
            check_at=None, P=16, group=1, cuda_cores=False, window=0):
    """Serial begin / append x layers / commit on the library and on the oracle model."""
    pool = pkv.Pool(layers, pool_pages, H, D, P, dtype_name(dtype), max_context, seed,
                    query_heads=H * group, cuda_cores=cuda_cores, window=window)
    req = pool.request()
    opool = OraclePool(layers, pool_pages, H, D, P, dtype, max_context=max_context, seed=seed,
                       query_heads=H * group, window=window)
    oreq = opool.request()
    errs = []
    for t in range(1, steps + 1):
        pos = req.begin_token()
        assert pos == oreq.begin_token() == t - 1
        if abort_at is not None and t == abort_at:
            for layer in range(layers - 1):
                q, k, v = _lane_tensors(seed, layer, H, pos, D, dtype, kseed=seed + 99, group=group)
                req.append_and_attend(layer, to_device(q), to_device(k),
                                      to_device(v))
                oreq.append_and_attend(layer, q, k, v, compute=False)
            req.abort_token()
            oreq.abort_token()
            assert req.length == oreq.length == t - 1
            assert req.page_table() == oreq.table
            assert pool.free_list() == list(opool.free)
            assert req.begin_token() == oreq.begin_token() == pos
        compute = check_at is None or t in check_at
        for layer in range(layers):
            q, k, v = _lane_tensors(seed, layer, H, pos, D, dtype, group=group)
            out = req.append_and_attend(layer, to_device(q), to_device(k),
                                        to_device(v))
            ref = oreq.append_and_attend(layer, q, k, v, compute=compute)
            if compute:
                errs.append(check_close(out.cpu().numpy(), ref, dtype, f"t={t} layer={layer}"))
        req.commit_token()
        oreq.commit_token()
        assert req.length == oreq.length == t
        assert req.page_table() == oreq.table
    assert pool.free_list() == list(opool.free)
    # every byte of the request's pages, in every layer, equals the oracle's pool
    used = torch.tensor(req.page_table(), dtype=torch.int64)
    for layer in range(layers):
        kd, vd = pool.kv_pages(layer)
        assert _host(kd[used.cuda()], dtype).tobytes() == opool.k[layer][used.numpy()].tobytes()
        assert _host(vd[used.cuda()], dtype).tobytes() == opool.v[layer][used.numpy()].tobytes()
    assert pool.check_device_status() == 0
    c = req.counters()
    assert c == {"committed_tokens": oreq.committed_tokens, "cache_appends": oreq.cache_appends,
                 "score_cells": oreq.score_cells}
    pool.close()
    return c, errs


def test_tiny_fixture_with_abort_and_retry():
    """1 request, 2 layers, H=2, d_h=2, pages of 16, pool of 4 pages, t = 1..4, abort at t=3."""
    w = workloads.tiny()
    c, errs = _serial(w.layers, w.H, w.D, F32, w.pool_pages, w.max_context, 4, w.seed, abort_at=3)
    assert c["score_cells"] == 4 * (1 + 2 + 3 + 4)
    assert c["cache_appends"] == 2 * 4


def test_tiny_fixture_counts_match_printed_values():
    c, _ = _serial(2, 2, 2, F32, 4, 64, 3, 0)
    assert c["score_cells"] == 24 and c["cache_appends"] == 6


@pytest.mark.parametrize("t", [128, 512, 2048])
def test_single_request_serial(t):
    """12 layers, H=12, d_h=64, fp32, 4096-page shuffled pool, serial appends to t."""
    checks = {1, 2, 15, 16, 17, 33, t // 2, t - 1, t}
    _, errs = _serial(12, 12, 64, F32, 4096, 2048, t, 1, check_at=checks)
    assert max(errs) <= FP32_ATOL


@pytest.mark.parametrize("H,D,dtype,window,t,group", [
    (4, 64, F32, 0, 900, 1),       # 57 tiles per lane: 56 workers, a cluster of 7 CTAs
    (4, 64, F32, 700, 900, 1),     # a window of 700 positions: 44-45 tiles, clusters of 5 CTAs
    (2, 128, BF16, 0, 520, 1),     # bf16 rows of 128: 33 tiles, a cluster of 4 CTAs
    (6, 64, F32, 0, 200, 1),       # 13 tiles: 8 workers inside one CTA
    # grouped-query pools on the tensor-core kernel (bf16, partials of G rows)
    (8, 128, BF16, 0, 520, 4),     # 33 tiles: a cluster of 4 CTAs per KV head
    (4, 64, BF16, 300, 700, 8),    # a window: 19-20 tiles, clusters of 2 CTAs
    (2, 128, BF16, 0, 200, 2),     # 13 tiles: 8 workers inside one CTA
    (2, 64, F32, 0, 4200, 1),      # 263 tiles: past 4 a worker, the global merge
    (2, 64, F32, 1000, 4200, 1),   # the same length in a window of 1000: clusters again
])
def test_single_request_lane_geometries(H, D, dtype, window, t, group):
    """Single requests whose lanes split over every worker count the launch picks:
    inside one CTA, and clusters of 2 to 7 CTAs (the two-level merge), with and
    without a sliding window, on both split kernels; checked against the oracle at
    lengths where the lane geometry changes."""
    checks = {1, 16, 17, 129, t // 2, t - 1, t}
    _, errs = _serial(2, H, D, dtype, 512, max(1024, t), t, 3, check_at=checks, window=window,
                      group=group)
    assert errs


def test_serial_bf16_and_page_size_32():
    _serial(3, 4, 128, BF16, 64, 200, 70, 5, abort_at=33, P=32)


@pytest.mark.parametrize("layers,dtype,H,t0", [(1, F32, 4, 0), (2, BF16, 4, 0), (12, F32, 12, 300)])
def test_back_to_back_tokens_without_host_copies(layers, dtype, H, t0):
    """Tokens issued back to back through the C ABI with every input already on the
    device, so each call's kernel is a dependent launch of the previous call's (no
    host copy between them breaks the chain): with one layer every kernel attends
    over the row the kernel just before it appended.  The page table, the lengths,
    every output and every appended byte equal the oracle model's.  t0 tokens go in
    first through the binding; the next 40 are checked."""
    import ctypes
    D, P, T, seed = 64, 16, 40, 23
    pool = pkv.Pool(layers, 128, H, D, P, dtype_name(dtype), 512, seed)
    req = pool.request()
    opool = OraclePool(layers, 128, H, D, P, dtype, max_context=512, seed=seed)
    oreq = opool.request()
    for t in range(t0):
        pos = req.begin_token()
        assert pos == oreq.begin_token()
        for layer in range(layers):
            q, k, v = _lane_tensors(seed, layer, H, pos, D, dtype)
            req.append_and_attend(layer, to_device(q), to_device(k), to_device(v))
            oreq.append_and_attend(layer, q, k, v, compute=False)
        req.commit_token()
        oreq.commit_token()
    host = [[_lane_tensors(seed, layer, H, t0 + i, D, dtype) for layer in range(layers)]
            for i in range(T)]
    qd = to_device(np.stack([[x[0] for x in row] for row in host]))   # [T][layers][H][D]
    kd = to_device(np.stack([[x[1] for x in row] for row in host]))
    vd = to_device(np.stack([[x[2] for x in row] for row in host]))
    out = torch.full((T, layers, H, D), float("nan"), device="cuda")
    torch.cuda.synchronize()
    lib, h = pkv.lib, req.handle
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    pos = ctypes.c_int64()

    def at(x, i, layer):
        return ctypes.c_void_p(x[i, layer].data_ptr())

    for i in range(T):
        assert lib.pkv_begin_token(h, ctypes.byref(pos)) == pkv.PKV_OK
        for layer in range(layers):
            assert lib.pkv_append_and_attend(h, layer, at(qd, i, layer), at(kd, i, layer),
                                             at(vd, i, layer), at(out, i, layer), stream) == pkv.PKV_OK
        assert lib.pkv_commit_token(h) == pkv.PKV_OK
    torch.cuda.synchronize()
    assert pool.check_device_status() == 0
    got = out.cpu().numpy()
    for i in range(T):
        assert oreq.begin_token() == t0 + i
        for layer in range(layers):
            q, k, v = host[i][layer]
            ref = oreq.append_and_attend(layer, q, k, v)
            check_close(got[i, layer], ref, dtype, f"token {t0 + i} layer {layer}")
        oreq.commit_token()
    assert req.length == oreq.length == t0 + T
    assert req.page_table() == oreq.table
    used = torch.tensor(req.page_table(), dtype=torch.int64)
    for layer in range(layers):
        kp, vp = pool.kv_pages(layer)
        assert _host(kp[used.cuda()], dtype).tobytes() == opool.k[layer][used.numpy()].tobytes()
        assert _host(vp[used.cuda()], dtype).tobytes() == opool.v[layer][used.numpy()].tobytes()
    req.close()
    pool.close()


# ------------------------------------------------------------------ batched --

def _batched_check(w, requests=None, heads=None, **kw):
    run = BatchedRun(w, **kw)
    try:
        assert run.tables.tolist() == run.otables.tolist()
        out = run.run().cpu().numpy()
        assert run.pool.check_device_status() == 0
        ref = run.oracle_out(requests, heads)
        got = np.stack([out[b, h] for (b, h) in ref])
        exp = np.stack(list(ref.values()))
        err = check_close(got, exp, w.dtype, w.name)
        reqs = range(w.B) if requests is None else requests
        for b in reqs:
            k, v = run.appended_rows(b)
            assert k.tobytes() == run.k_new[b].tobytes() and v.tobytes() == run.v_new[b].tobytes()
        return run, err
    finally:
        run.close()


@pytest.mark.parametrize("dtype", [F32, BF16])
def test_batched_decode_full_config(dtype):
    """64 requests, H=32, d_h=128, t ~ U{1..4096}, 32768-page shuffled pool: every lane."""
    _batched_check(workloads.batched(dtype))


def test_ragged_fragmented_pool_sampled():
    """256 requests, lognormal lengths, 600k-page pool after 10k lease/release cycles:
    the longest, the shortest and 30 random requests, all heads."""
    w = workloads.ragged()
    order = np.argsort(w.seq_lens)
    rng = np.random.default_rng(0)
    sample = sorted(set([int(order[0]), int(order[-1]), int(order[len(order) // 2])] +
                        rng.choice(w.B, 30, replace=False).tolist()))
    _batched_check(w, requests=sample)


def test_long_context_sampled():
    """16 requests x 131072 tokens, H=8, d_h=128, bf16: 3 requests, all heads."""
    _batched_check(workloads.long_context(), requests=[0, 7, 15])


# --------------------------------------------------------------- edge cases --

@pytest.mark.parametrize("dtype", [F32, BF16])
def test_ragged_tails_and_single_tokens(dtype):
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 47, 48, 49, 1, 64, 255, 256, 257]
    _batched_check(make_workload("tails", lens, 3, 64, dtype=dtype, seed=3))


def test_all_single_token_requests():
    w = make_workload("ones", [1] * 37, 4, 32, dtype=BF16, seed=4)
    run, _ = _batched_check(w)


@pytest.mark.parametrize("D,dtype", [(2, F32), (4, F32), (8, F32), (16, BF16), (32, F32),
                                     (64, BF16), (128, F32), (256, BF16), (2, BF16)])
def test_head_widths(D, dtype):
    _batched_check(make_workload(f"d{D}", [1, 40, 100, 16, 77], 2, D, dtype=dtype, seed=D))


@pytest.mark.parametrize("P", [32, 64])
def test_page_sizes(P):
    _batched_check(make_workload(f"p{P}", [1, 31, 33, 64, 65, 200], 2, 64, P=P, dtype=F32, seed=P))


def test_contiguous_single_page_layout_equals_paged():
    """One max-context page per request (page_size = max_context) gives the paged result."""
    lens = [37, 256, 5, 129]
    a = BatchedRun(make_workload("paged", lens, 2, 64, P=16, dtype=F32, seed=8))
    b = BatchedRun(make_workload("contig", lens, 2, 64, P=256, dtype=F32, seed=8, max_context=256))
    try:
        assert b.tables.shape[1] == 1
        oa, ob = a.run().cpu().numpy(), b.run().cpu().numpy()
        assert np.abs(oa - ob).max() <= 2e-6
        ref = a.oracle_out()
        check_close(np.stack([ob[k] for k in ref]), np.stack(list(ref.values())), F32, "contig")
    finally:
        a.close()
        b.close()


def test_more_workers_than_tiles():
    """A loose max_seq_len gives far more workers than tiles (empty workers)."""
    _batched_check(make_workload("few", [40, 3], 1, 64, dtype=F32, seed=9, max_context=8192),
                   max_seq_len=8192)


def test_wide_page_table_rows_and_side_stream():
    s = torch.cuda.Stream()
    w = make_workload("stream", [300, 20, 1000], 4, 128, dtype=BF16, seed=10)
    with torch.cuda.stream(s):
        _batched_check(w, page_table_pad=5, stream=s)
    torch.cuda.synchronize()


def test_repeated_calls_are_deterministic():
    w = make_workload("rep", [1000, 17, 4000, 2], 8, 128, dtype=BF16, seed=11)
    run = BatchedRun(w)
    try:
        a = run.run().clone()
        b = run.run().clone()
        assert torch.equal(a, b)
    finally:
        run.close()


def test_bad_lengths_and_page_ids_set_error_bits():
    w = make_workload("bad", [20, 50, 7], 2, 64, dtype=F32, seed=12)
    run = BatchedRun(w)
    try:
        good = run.run().cpu().numpy()
        assert run.pool.check_device_status() == 0
        lens = run.dev["lens"].clone()
        run.dev["lens"][0] = 0                       # t < 1
        run.run()
        assert run.pool.device_status_bits() & pkv.PKV_DEVERR_SEQ_LEN
        run.dev["lens"].copy_(lens)
        run.dev["lens"][1] = run.max_seq_len + 1     # t > max_seq_len
        run.run()
        assert run.pool.device_status_bits() & pkv.PKV_DEVERR_SEQ_LEN
        run.dev["lens"].copy_(lens)
        saved = run.dev["tables"][1, 1].item()
        run.dev["tables"][1, 1] = run.pool.pages     # page id out of range
        out = run.run().cpu().numpy()
        assert run.pool.device_status_bits() & pkv.PKV_DEVERR_PAGE_ID
        assert np.array_equal(out[0], good[0]) and np.array_equal(out[2], good[2])
        run.dev["tables"][1, 1] = saved
        out = run.run().cpu().numpy()
        assert run.pool.check_device_status() == 0
        assert np.abs(out - good).max() == 0
    finally:
        run.close()


def test_argument_errors_change_nothing():
    w = make_workload("args", [10, 20], 2, 64, dtype=F32, seed=13)
    run = BatchedRun(w)
    try:
        d = run.dev
        import ctypes
        st = pkv.lib.pkv_paged_decode_attention(
            run.pool.handle, 0, 2, ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(d["k"].data_ptr()),
            ctypes.c_void_p(d["v"].data_ptr()), ctypes.c_void_p(d["tables"].data_ptr()),
            d["tables"].shape[1], ctypes.c_void_p(d["lens"].data_ptr()), 20,
            ctypes.c_void_p(run.out.data_ptr()), ctypes.c_void_p(run.ws.data_ptr()), 16, None)
        assert st == pkv.PKV_ERR_INVALID_ARGUMENT
        st = pkv.lib.pkv_paged_decode_attention(run.pool.handle, 0, 0, None, None, None, None, 1,
                                                None, 1, None, None, 0, None)
        assert st == pkv.PKV_OK
        st = pkv.lib.pkv_paged_decode_attention(run.pool.handle, 1, 2, None, None, None, None, 1,
                                                None, 1, None, None, 0, None)
        assert st == pkv.PKV_ERR_INVALID_ARGUMENT
        assert torch.isnan(run.out).all()
        with pytest.raises(pkv.PkvError) as e:
            pkv.Pool(1, 4, 2, 96, 16, "bf16", 64)
        assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
        with pytest.raises(pkv.PkvError) as e:
            pkv.Pool(1, 4, 2, 64, 8, "bf16", 64)
        assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    finally:
        run.close()


# ------------------------------------------------------------ grouped query --

@pytest.mark.parametrize("group,D,dtype", [(2, 64, F32), (4, 64, BF16), (8, 64, F32),
                                           (2, 128, BF16), (4, 128, F32), (8, 128, BF16),
                                           (8, 128, F32)])
def test_gqa_batched(group, D, dtype):
    lens = [1, 16, 17, 300, 1000, 33, 2048, 5]
    _batched_check(make_workload(f"gqa{group}", lens, 2, D, dtype=dtype, seed=40 + group,
                                 group=group))


# fp32 pools with several query heads per KV head run the tensor-core kernel on
# split tf32 products (each operand as its tf32 rounding plus the rounding of the
# rest; all four cross products), held to the fp32 bar; PKV_POOL_CUDA_CORES keeps
# the CUDA-core kernel for the same geometry.

@pytest.mark.parametrize("group,D", [(2, 64), (8, 128)])
def test_gqa_fp32_cuda_core_kernel(group, D):
    lens = [1, 16, 17, 300, 1000, 33, 2048, 5]
    _batched_check(make_workload(f"cc32_{group}", lens, 2, D, dtype=F32, seed=140 + group,
                                 group=group), cuda_cores=True)


def test_fp32_tensor_core_and_cuda_core_kernels_agree():
    w = make_workload("agree32", [1, 15, 16, 17, 500, 4096, 33], 2, 128, dtype=F32, seed=62,
                      group=8)
    a, b = BatchedRun(w), BatchedRun(w, cuda_cores=True)
    try:
        assert a.pool.kernel_name() == "split_decode_mma_kernel<f32,128,8>"
        assert b.pool.kernel_name() == "split_decode_kernel<f32,128,8>"
        oa, ob = a.run().cpu().numpy(), b.run().cpu().numpy()
        assert np.abs(oa - ob).max() < 4e-6
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("group,D,P,window", [(4, 128, 32, 0), (8, 64, 64, 0), (2, 128, 16, 100),
                                              (8, 128, 16, 4000)])
def test_gqa_fp32_tensor_core_pages_and_windows(group, D, P, window):
    lens = [1, 15, 16, 17, 64, 65, 500, 1999, 4096]
    _batched_check(make_workload(f"tc32_{group}_{P}_{window}", lens, 2, D, P=P, dtype=F32,
                                 seed=150 + group + P, group=group, window=window))


def test_gqa_fp32_tensor_core_serial_with_abort():
    c, _ = _serial(2, 2, 128, F32, 64, 300, 70, 14, abort_at=33, P=32, group=4)
    assert c["score_cells"] == 2 * 8 * sum(range(1, 71))


def test_gqa_full_config_every_lane():
    """64 requests, 8 KV heads x 8 query heads, d_h=128, bf16, t ~ U{1..8192}."""
    _batched_check(workloads.gqa(8))


def test_gqa_serial_with_abort():
    c, _ = _serial(2, 2, 64, BF16, 64, 200, 40, 7, abort_at=17, group=4)
    assert c["score_cells"] == 2 * 8 * sum(range(1, 41))


def test_gqa_more_workers_than_tiles():
    _batched_check(make_workload("gqa_few", [40, 3], 1, 128, dtype=BF16, seed=46, group=8,
                                 max_context=8192), max_seq_len=8192)


def test_gqa_geometry_errors():
    with pytest.raises(pkv.PkvError) as e:
        pkv.Pool(1, 8, 2, 64, 16, "bf16", 64, query_heads=6)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    with pytest.raises(pkv.PkvError) as e:
        pkv.Pool(1, 8, 4, 64, 16, "bf16", 64, query_heads=6)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARGUMENT
    with pytest.raises(pkv.PkvError) as e:
        pkv.Pool(1, 8, 2, 32, 16, "bf16", 64, query_heads=4)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED


# --------------------------------------------------------------- multi-query --
# 16 .. 128 query heads per KV head (down to a single KV head): decode runs them as
# lanes of 8 query heads, 2^s lanes per KV head, each reading the KV head's pages.

@pytest.mark.parametrize("group,H,D,dtype,cc", [(16, 2, 128, BF16, False), (32, 1, 128, BF16, False),
                                                (64, 1, 64, BF16, False), (128, 1, 128, BF16, False),
                                                (16, 2, 64, F32, False), (32, 2, 128, F32, False),
                                                (16, 2, 128, BF16, True)])
def test_mqa_batched(group, H, D, dtype, cc):
    lens = [1, 16, 17, 300, 1000, 33, 2048, 5]
    _batched_check(make_workload(f"mqa{group}", lens, H, D, dtype=dtype, seed=80 + group,
                                 group=group), cuda_cores=cc)


def test_mqa_window_and_few_tiles():
    _batched_check(make_workload("mqawin", [1, 2, 40, 129, 700, 3000], 2, 128, dtype=BF16,
                                 seed=93, group=16, window=200))
    _batched_check(make_workload("mqa_few", [40, 3], 1, 128, dtype=BF16, seed=94, group=32,
                                 max_context=8192), max_seq_len=8192)


def test_mqa_serial_with_abort():
    c, _ = _serial(2, 2, 128, BF16, 64, 200, 40, 7, abort_at=17, group=16)
    assert c["score_cells"] == 2 * 32 * sum(range(1, 41))
    _serial(2, 1, 64, F32, 64, 200, 30, 8, abort_at=9, group=32)


def test_mqa_geometry():
    for g in (16, 32, 64, 128):
        with pkv.Pool(1, 8, 1, 128, 16, "bf16", 64, query_heads=g) as p:
            assert p.query_heads == g and p.tensor_cores
    for g in (12, 24, 256):
        with pytest.raises(pkv.PkvError) as e:
            pkv.Pool(1, 8, 1, 128, 16, "bf16", 64, query_heads=g)
        assert e.value.status == pkv.PKV_ERR_UNSUPPORTED


# ---------------------------------------- tensor-core and CUDA-core kernels --
# bf16 grouped-query pools at head width 64 or 128 run the tensor-core kernel by
# default; PKV_POOL_CUDA_CORES selects the CUDA-core kernel for the same geometry.

def test_kernel_selection():
    def pool(**kw):
        return pkv.Pool(1, 8, 2, kw.pop("D", 128), 16, kw.pop("dtype", "bf16"), 64, **kw)
    with pool(query_heads=16) as p:
        assert p.tensor_cores and p.kernel_name() == "split_decode_mma_kernel<bf16,128,8>"
    with pool(query_heads=32) as p:
        assert p.tensor_cores and p.kernel_name() == "split_decode_mma_kernel<bf16,128,16>"
    with pool(query_heads=64, D=64) as p:
        assert p.tensor_cores and p.kernel_name() == "split_decode_mma_kernel<bf16,64,16>"
    with pool(query_heads=16, cuda_cores=True) as p:
        assert not p.tensor_cores
    with pool() as p:
        assert not p.tensor_cores
    with pool(query_heads=4, dtype="f32") as p:
        assert p.tensor_cores and p.kernel_name() == "split_decode_mma_kernel<f32,128,2>"
    with pool(query_heads=64, dtype="f32", D=64) as p:
        assert p.tensor_cores and p.kernel_name() == "split_decode_mma_kernel<f32,64,8>"
    with pool(dtype="f32") as p:
        assert not p.tensor_cores
    with pool(query_heads=4, dtype="f32", cuda_cores=True) as p:
        assert not p.tensor_cores and p.kernel_name() == "split_decode_kernel<f32,128,2>"


@pytest.mark.parametrize("group,D", [(2, 64), (4, 128), (8, 128)])
def test_gqa_cuda_core_kernel(group, D):
    lens = [1, 16, 17, 300, 1000, 33, 2048, 5]
    _batched_check(make_workload(f"cc{group}", lens, 2, D, dtype=BF16, seed=50 + group,
                                 group=group), cuda_cores=True)


def test_serial_bf16_gqa_cuda_core_kernel_with_abort():
    _serial(3, 4, 128, BF16, 64, 200, 70, 5, abort_at=33, P=32, group=2, cuda_cores=True)


def test_serial_bf16_tensor_core_gqa_page_size_64():
    _serial(2, 2, 128, BF16, 64, 300, 90, 9, abort_at=65, P=64, group=8)


def test_tensor_core_and_cuda_core_kernels_agree():
    w = make_workload("agree", [1, 15, 16, 17, 500, 4096, 33], 4, 128, dtype=BF16, seed=60, group=4)
    a, b = BatchedRun(w), BatchedRun(w, cuda_cores=True)
    try:
        oa, ob = a.run().cpu().numpy(), b.run().cpu().numpy()
        rel = np.abs(oa - ob).max(axis=-1) / np.maximum(np.abs(ob).max(axis=-1), 1e-6)
        assert rel.max() < 1e-4
    finally:
        a.close()
        b.close()



# 16-query lanes: groups of 16 and more run on the tensor-core kernel as lanes of 16
# query heads (two MMA rows per fragment lane); the CUDA-core kernel runs them as
# lanes of 8.  Page sizes 32 and 64 put several tiles in a page.

@pytest.mark.parametrize("group,H,D,P,window", [(16, 2, 128, 32, 0), (16, 1, 64, 64, 0),
                                                (32, 2, 64, 16, 77), (16, 3, 128, 64, 300)])
def test_wide_lanes_page_sizes(group, H, D, P, window):
    lens = [1, 15, 16, 17, 64, 65, 500, 1999, 4096]
    _batched_check(make_workload(f"wide{group}_{P}", lens, H, D, P=P, dtype=BF16,
                                 seed=110 + group + P, group=group, window=window))


def test_wide_lanes_agree_with_cuda_core_lanes_of_8():
    w = make_workload("wide_agree", [1, 15, 16, 17, 500, 4096, 33], 2, 128, dtype=BF16, seed=61,
                      group=32)
    a, b = BatchedRun(w), BatchedRun(w, cuda_cores=True)
    try:
        assert a.pool.kernel_name() == "split_decode_mma_kernel<bf16,128,16>"
        assert b.pool.kernel_name() == "split_decode_kernel<bf16,128,8>"
        oa, ob = a.run().cpu().numpy(), b.run().cpu().numpy()
        rel = np.abs(oa - ob).max(axis=-1) / np.maximum(np.abs(ob).max(axis=-1), 1e-6)
        assert rel.max() < 1e-4
    finally:
        a.close()
        b.close()


def test_wide_lanes_serial_page_size_32_with_abort():
    _serial(2, 1, 64, BF16, 64, 300, 70, 12, abort_at=33, P=32, group=16)

# ----------------------------------------------------------- sliding window --

@pytest.mark.parametrize("window,dtype,group", [(1, F32, 1), (16, BF16, 1), (17, F32, 1),
                                                (100, BF16, 1), (64, BF16, 4), (333, BF16, 8),
                                                (5000, BF16, 2)])
def test_window_batched(window, dtype, group):
    lens = [1, 2, 16, 17, 33, 100, 101, 300, 1000, 4097]
    D = 128 if group > 1 else 64
    _batched_check(make_workload(f"win{window}", lens, 2, D, dtype=dtype, seed=70 + window,
                                 group=group, window=window))


def test_window_cuda_core_kernel_gqa():
    lens = [5, 16, 17, 300, 1000, 2049]
    _batched_check(make_workload("wincc", lens, 2, 128, dtype=BF16, seed=77, group=4, window=129),
                   cuda_cores=True)


def test_window_full_config_every_lane():
    """64 requests, t ~ U{1..32768}, window 4096, 8 KV heads x 4 query heads."""
    _batched_check(workloads.sliding_window())


def test_window_serial_with_abort():
    c, _ = _serial(2, 2, 64, F32, 64, 300, 60, 8, abort_at=40, window=20)
    assert c["score_cells"] == 2 * 2 * sum(min(t, 20) for t in range(1, 61))


def test_window_serial_gqa_tensor_cores():
    _serial(2, 2, 128, BF16, 64, 300, 50, 9, group=8, window=33)


# ----------------------------------------------------------- prefix sharing --

def _token(seed, layers, H, pos, D, dtype, group=1):
    return [_lane_tensors(seed, layer, H, pos, D, dtype, group=group) for layer in range(layers)]


@pytest.mark.parametrize("dtype,group,fork_at", [(F32, 1, 37), (BF16, 4, 48), (BF16, 1, 20)])
def test_fork_then_divergent_decodes(dtype, group, fork_at):
    """Parent and child share the prefix; each then decodes its own tokens.  The
    partially filled shared page is copied on the first write; outputs, tables,
    references and every used page's bytes match the oracle model."""
    layers, H, D, P = 2, 2, 128 if group > 1 else 64, 16
    pool = pkv.Pool(layers, 64, H, D, P, dtype_name(dtype), 512, 3, query_heads=H * group)
    opool = OraclePool(layers, 64, H, D, P, dtype, max_context=512, seed=3, query_heads=H * group)
    parent, oparent = pool.request(), opool.request()

    def step(req, oreq, seed, check=True):
        pos = req.begin_token()
        assert oreq.begin_token() == pos
        for layer, (q, k, v) in enumerate(_token(seed, layers, H, pos, D, dtype, group)):
            out = req.append_and_attend(layer, to_device(q), to_device(k), to_device(v))
            ref = oreq.append_and_attend(layer, q, k, v)
            if check:
                check_close(out.cpu().numpy(), ref, dtype, f"pos={pos} layer={layer}")
        req.commit_token()
        oreq.commit_token()

    for _ in range(fork_at):
        step(parent, oparent, 1, check=False)
    child, ochild = parent.fork(), oparent.fork()
    assert child.length == parent.length == fork_at
    for i in range(20):
        step(parent, oparent, 100)
        step(child, ochild, 200)
        if i == 3:   # abort a token of the child, then go on
            child.begin_token()
            ochild.begin_token()
            child.abort_token()
            ochild.abort_token()
    for r, o in ((parent, oparent), (child, ochild)):
        assert r.page_table() == o.table and r.length == o.length
    assert pool.free_list() == list(opool.free)
    assert [pool.page_refs(i) for i in range(64)] == opool.refs
    used = sorted(set(parent.page_table()) | set(child.page_table()))
    idx = torch.tensor(used, dtype=torch.int64)
    for layer in range(layers):
        kd, vd = pool.kv_pages(layer)
        assert _host(kd[idx.cuda()], dtype).tobytes() == opool.k[layer][used].tobytes()
        assert _host(vd[idx.cuda()], dtype).tobytes() == opool.v[layer][used].tobytes()
    assert pool.check_device_status() == 0
    pool.close()



def test_shared_prompt_batched_every_lane():
    """64 requests forked from one 8192-token prompt (shared pages), each with its own
    suffix, decoded in one batched call: every lane against the oracle."""
    run, _ = _batched_check(workloads.shared_prompt())


def test_shared_prompt_small_mixed():
    w = workloads.shared_prompt(seed=8, B=5, prefix=64, suffix_max=40)
    _batched_check(w)
