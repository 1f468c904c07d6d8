"""Failure injection on device pools, through the C ABI (GPU).

Host side: a layer call armed to fail ("Incremental Serving", section "Request
flow", step 4: after a failure, abort leaves the visible length unchanged) is
followed by pkv_abort_token; lengths, tables, page references, the free list,
counters and every visible K/V byte then equal the oracle model's after the same
begin and abort, and a retry gives the oracle's outputs.

Device side: a split worker arms its first stage's barrier without issuing the
copy, so its bounded wait (a few ms here) runs out.  The launch ends by itself,
the pool's error word holds PKV_DEVERR_TIMEOUT, the other lanes' rows are
right, and the next call on the same context matches the oracle.  Nothing
faults or hangs: the wait is bounded and the worker lets the copies it issued
land before it returns.
"""
import time

import numpy as np
import pytest
import torch

import paged_kv_cache_decode_gb300 as pkv
import synth
from oracle.model import OraclePool
from synth import BF16, F32
from synth.device import to_device
from tests._gpu import BatchedRun, check_close, make_workload

pytestmark = pytest.mark.gpu

WAIT_NS = 3_000_000          # 3 ms: the armed worker's wait runs out after this


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _rows(rng, shape, dtype):
    x = rng.standard_normal(shape).astype(np.float32)
    return x if dtype == F32 else synth.f32_to_bf16(x)


def _q32(x):
    return synth.bf16_to_f32(x) if x.dtype == np.uint16 else x


def _host(t, dtype):
    t = t.cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if dtype == BF16 else t.numpy()


def _same_state(pool, opool, reqs, oreqs):
    for r, o in zip(reqs, oreqs):
        assert r.page_table() == o.table and r.length == o.length
        c = r.counters()
        assert (c["committed_tokens"], c["cache_appends"], c["score_cells"]) == (
            o.committed_tokens, o.cache_appends, o.score_cells)
    assert pool.free_list() == list(opool.free)
    assert [pool.page_refs(x) for x in range(opool.pages)] == opool.refs


def _visible_bytes_equal(pool, opool, reqs, oreqs, dtype):
    for layer in range(opool.layers):
        kd, vd = pool.kv_pages(layer)
        for r, o in zip(reqs, oreqs):
            for j in range(o.length):
                pg, slot = o.table[j // opool.P], j % opool.P
                assert _host(kd[pg, :, slot], dtype).tobytes() == opool.k[layer][pg, :, slot].tobytes()
                assert _host(vd[pg, :, slot], dtype).tobytes() == opool.v[layer][pg, :, slot].tobytes()


def _token(rng, r, o, layers, HQ, H, D, dtype, upto=None):
    """Append every layer (or layers < upto) of the pending token on both sides."""
    errs = []
    for layer in range(layers if upto is None else upto):
        q = rng.standard_normal((HQ, D)).astype(np.float32)
        k, v = _rows(rng, (H, D), dtype), _rows(rng, (H, D), dtype)
        out = r.append_and_attend(layer, to_device(q), to_device(k), to_device(v))
        ref = o.append_and_attend(layer, q, k, v)
        errs.append(check_close(out.cpu().numpy(), ref, dtype, f"layer {layer}"))
    return errs


@pytest.mark.parametrize("dtype,D,G", [(F32, 64, 1), (BF16, 128, 4)])
def test_layer_failure_mid_token_then_abort(dtype, D, G):
    layers, H, P, pages, maxc = 3, 2, 16, 12, 96
    rng = np.random.default_rng(3)
    pool = pkv.Pool(layers, pages, H, D, P, "f32" if dtype == F32 else "bf16", maxc, 4,
                    query_heads=H * G)
    opool = OraclePool(layers, pages, H, D, P, dtype, max_context=maxc, seed=4, query_heads=H * G)
    try:
        r, o = pool.request(), opool.request()
        for _ in range(16):                       # 16 committed: the next token starts a page
            r.begin_token()
            o.begin_token()
            _token(rng, r, o, layers, H * G, H, D, dtype)
            r.commit_token()
            o.commit_token()
        r.begin_token()
        o.begin_token()
        _token(rng, r, o, layers, H * G, H, D, dtype, upto=1)
        pool.inject_fault(pkv.PKV_INJECT_LAYER, 1)
        q = torch.zeros((H * G, D), device="cuda")
        kv = torch.zeros((H, D), device="cuda",
                         dtype=torch.float32 if dtype == F32 else torch.bfloat16)
        with pytest.raises(pkv.PkvError) as e:
            r.append_and_attend(1, q, kv, kv)
        assert e.value.status == pkv.PKV_ERR_CUDA and "injected" in str(e.value)
        with pytest.raises(pkv.PkvError) as e:
            r.commit_token()                      # layers 1 and 2 did not run
        assert e.value.status == pkv.PKV_ERR_BAD_STATE
        r.abort_token()
        o.abort_token()
        assert r.length == 16
        _same_state(pool, opool, [r], [o])
        _visible_bytes_equal(pool, opool, [r], [o], dtype)
        # the retry after the abort is exact
        r.begin_token()
        o.begin_token()
        _token(rng, r, o, layers, H * G, H, D, dtype)
        r.commit_token()
        o.commit_token()
        _same_state(pool, opool, [r], [o])
        _visible_bytes_equal(pool, opool, [r], [o], dtype)
        assert pool.check_device_status() == 0
        r.close()
    finally:
        pool.close()


@pytest.mark.parametrize("dtype,D", [(F32, 64), (BF16, 64)])
def test_layer_failure_in_chunk_with_copy_on_write(dtype, D):
    """A forked request's chunk (a copy-on-write page and a fresh one) fails on its
    second layer; abort restores the shared page, the sharer's bytes are untouched."""
    layers, H, G, P, pages, maxc = 2, 2, 2, 16, 16, 128
    rng = np.random.default_rng(8)
    pool = pkv.Pool(layers, pages, H, D, P, "f32" if dtype == F32 else "bf16", maxc, 6,
                    query_heads=H * G)
    opool = OraclePool(layers, pages, H, D, P, dtype, max_context=maxc, seed=6, query_heads=H * G)
    try:
        a, oa = pool.request(), opool.request()
        for _ in range(20):
            a.begin_token()
            oa.begin_token()
            _token(rng, a, oa, layers, H * G, H, D, dtype)
            a.commit_token()
            oa.commit_token()
        b, ob = a.fork(), oa.fork()
        reqs, oreqs = [a, b], [oa, ob]
        _same_state(pool, opool, reqs, oreqs)
        n = 20                                    # positions 20..39: page 1 (shared) and page 2
        b.begin_chunk(n)
        ob.begin_chunk(n)
        q = _rows(rng, (n, H * G, D), dtype)
        k, v = _rows(rng, (n, H, D), dtype), _rows(rng, (n, H, D), dtype)
        out = b.prefill_chunk(0, to_device(q), to_device(k), to_device(v))
        ref = ob.prefill_chunk(0, _q32(q), k, v)
        check_close(out.cpu().numpy(), ref, dtype, "chunk layer 0")
        pool.inject_fault(pkv.PKV_INJECT_LAYER, 1)
        with pytest.raises(pkv.PkvError) as e:
            b.prefill_chunk(1, to_device(q), to_device(k), to_device(v))
        assert e.value.status == pkv.PKV_ERR_CUDA
        b.abort_token()
        ob.abort_token()
        _same_state(pool, opool, reqs, oreqs)
        _visible_bytes_equal(pool, opool, reqs, oreqs, dtype)
        b.begin_chunk(n)
        ob.begin_chunk(n)
        for layer in range(layers):
            out = b.prefill_chunk(layer, to_device(q), to_device(k), to_device(v))
            ref = ob.prefill_chunk(layer, _q32(q), k, v)
            check_close(out.cpu().numpy(), ref, dtype, f"retry layer {layer}")
        b.commit_token()
        ob.commit_token()
        _same_state(pool, opool, reqs, oreqs)
        _visible_bytes_equal(pool, opool, reqs, oreqs, dtype)
        assert pool.check_device_status() == 0
        for r in reqs:
            r.close()
    finally:
        pool.close()


def test_lease_failure_on_a_device_pool():
    layers, H, D, P = 2, 2, 64, 16
    rng = np.random.default_rng(9)
    pool = pkv.Pool(layers, 8, H, D, P, "f32", 64, 2)
    opool = OraclePool(layers, 8, H, D, P, F32, max_context=64, seed=2)
    try:
        r, o = pool.request(), opool.request()
        for _ in range(16):
            r.begin_token()
            o.begin_token()
            _token(rng, r, o, layers, H, H, D, F32)
            r.commit_token()
            o.commit_token()
        pool.inject_fault(pkv.PKV_INJECT_LEASE, 1)
        with pytest.raises(pkv.PkvError) as e:
            r.begin_token()                       # position 16 needs a page
        assert e.value.status == pkv.PKV_ERR_OUT_OF_PAGES
        _same_state(pool, opool, [r], [o])
        r.begin_token()
        o.begin_token()
        _token(rng, r, o, layers, H, H, D, F32)
        r.commit_token()
        o.commit_token()
        _same_state(pool, opool, [r], [o])
        _visible_bytes_equal(pool, opool, [r], [o], F32)
        r.close()
    finally:
        pool.close()


def _oracle_array(run):
    ref = run.oracle_out()
    w = run.w
    return np.stack([np.stack([ref[(b, h)] for h in range(w.HQ)]) for b in range(w.B)])


@pytest.mark.parametrize("dtype,group", [(BF16, 1), (F32, 1), (BF16, 8)])
def test_device_wait_runs_out_and_the_context_stays_usable(dtype, group):
    """Worker 0 covers the first few tiles of request 0's first lane only (request 0
    is long, every worker takes >= 4 tiles); those rows are unspecified, every other
    row is right, and a clean call afterwards is right everywhere."""
    lens = [4096, 700, 33, 1, 2500, 16, 17, 1200]
    run = BatchedRun(make_workload("fault", lens, 4, 128, dtype=dtype, seed=51, group=group))
    try:
        orc = _oracle_array(run)
        run.pool.inject_fault(pkv.PKV_INJECT_DEVICE_WAIT, 0, WAIT_NS)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        out = run.run()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        bits = run.pool.device_status_bits()
        assert bits & pkv.PKV_DEVERR_TIMEOUT, bits
        assert dt < 2.0, f"the faulted launch took {dt:.3f} s"
        got = out.cpu().numpy()
        check_close(got[1:], orc[1:], dtype, "rows the armed worker does not feed")
        # the context is usable and the hook is spent: a clean call is right everywhere
        out = run.run()
        assert run.pool.check_device_status() == 0
        check_close(out.cpu().numpy(), orc, dtype, "after the timeout")
    finally:
        run.close()


def test_device_wait_in_a_single_request_token():
    """The transactional path: the first layer's launch loses its first tile's copy;
    the token is aborted and retried, and the retry matches the oracle."""
    layers, H, D, P = 2, 4, 64, 16
    rng = np.random.default_rng(12)
    pool = pkv.Pool(layers, 64, H, D, P, "f32", 1024, 7)
    opool = OraclePool(layers, 64, H, D, P, F32, max_context=1024, seed=7)
    try:
        r, o = pool.request(), opool.request()
        for _ in range(300):
            r.begin_token()
            o.begin_token()
            for layer in range(layers):
                q = rng.standard_normal((H, D)).astype(np.float32)
                k = rng.standard_normal((H, D)).astype(np.float32)
                v = rng.standard_normal((H, D)).astype(np.float32)
                r.append_and_attend(layer, to_device(q), to_device(k), to_device(v))
                o.append_and_attend(layer, q, k, v, compute=False)
            r.commit_token()
            o.commit_token()
        assert pool.check_device_status() == 0
        pool.inject_fault(pkv.PKV_INJECT_DEVICE_WAIT, 0, WAIT_NS)
        r.begin_token()
        o.begin_token()
        zq = torch.zeros((H, D), device="cuda")
        for layer in range(layers):
            r.append_and_attend(layer, zq, zq, zq)
        bits = pool.device_status_bits()
        assert bits & pkv.PKV_DEVERR_TIMEOUT, bits
        r.abort_token()
        o.abort_token()
        _same_state(pool, opool, [r], [o])
        r.begin_token()
        o.begin_token()
        _token(rng, r, o, layers, H, H, D, F32)
        r.commit_token()
        o.commit_token()
        _same_state(pool, opool, [r], [o])
        _visible_bytes_equal(pool, opool, [r], [o], F32)
        assert pool.check_device_status() == 0
        r.close()
    finally:
        pool.close()
