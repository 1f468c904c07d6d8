"""Batched prefill on the device vs the fp64 oracle, through the C ABI.

Bar: bit-exact K/V rows written into the pages; normwise relative error per
(token, query head) row <= PREFILL_RTOL, the bf16-storage bar of decode.  q, k
and v are the pool's bf16 values (the oracle reads the same bits); the tensor
cores multiply V by the softmax weights split into bf16 hi + lo, which carries
each weight to about 2^-16 relative, so the error left is that of fp32
accumulation and the exp2 approximation, far inside the bar.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_decode_gb300 as pkv
from synth import workloads
from tests._gpu import PrefillRun, make_prefill

pytestmark = pytest.mark.gpu

PREFILL_RTOL = 5e-3


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _normwise(out: np.ndarray, ref: np.ndarray) -> float:
    num = np.abs(out - ref).max(axis=-1)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-6)
    return float((num / den).max()) if out.size else 0.0


CASES = {
    # name: (cached, new, H, D, group, P, window)
    "d128_mha": ([0, 37, 300], [1, 50, 200], 2, 128, 1, 16, 0),
    "d64_gqa4": ([0, 129, 1000], [100, 33, 64], 2, 64, 4, 16, 0),
    "d128_gqa8_window": ([50, 400], [300, 16], 1, 128, 8, 16, 100),
    "d128_gqa2_page32": ([17], [259], 2, 128, 2, 32, 0),
    "d64_mha_long": ([2000], [130], 1, 64, 1, 16, 0),
    "empty_request": ([10, 5, 0], [0, 20, 0], 2, 128, 2, 16, 0),
    "d64_gqa8_window_ragged": ([0, 3, 700], [129, 255, 1], 2, 64, 8, 64, 33),
    # multi-query: a query tile is 128/G tokens x G heads
    "d128_mqa16": ([0, 45, 333], [70, 9, 130], 2, 128, 16, 16, 0),
    "d128_mqa32_window": ([100, 7], [41, 64], 1, 128, 32, 16, 50),
    "d64_mqa64": ([20], [23], 1, 64, 64, 16, 0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_oracle(name):
    cached, new, H, D, G, P, W = CASES[name]
    w = make_prefill(name, cached, new, H, D, group=G, P=P, window=W, seed=41)
    run = PrefillRun(w)
    try:
        out = run.run().cpu().numpy()
        torch.cuda.synchronize()
        assert run.pool.check_device_status() == 0
        worst = 0.0
        for b in range(w.B):
            nb = int(w.new_tokens[b])
            if nb == 0:
                continue
            got = out[run.cu[b]:run.cu[b + 1]]
            assert np.isfinite(got).all(), f"request {b}: non-finite output"
            err = _normwise(got, run.oracle_out(b))
            worst = max(worst, err)
            for i in range(nb):
                k, v = run.chunk_rows(b, i)
                x = int(run.cu[b]) + i
                assert np.array_equal(k, run.k_new[x]) and np.array_equal(v, run.v_new[x])
        print(f"{name}: worst normwise error {worst:.2e}")
        assert worst <= PREFILL_RTOL
    finally:
        run.close()


def test_prefill_v_far_from_unit_scale():
    """V rows far from unit scale: chunk rows scaled by 2^20 in some key tiles of
    request 0 (next to unscaled rows of the same tiles), and one request whose every
    V row is scaled by 2^-20.  Every row stays inside the bar: the weights carry
    their relative precision whatever V's scale.  Powers of two keep the bf16
    values exact."""
    import synth
    from synth.device import to_device
    w = make_prefill("v_range", [0, 200, 0], [300, 130, 257], 2, 128, group=4, seed=44)
    run = PrefillRun(w)
    try:
        v = synth.bf16_to_f32(run.v_new).copy()
        c = run.cu
        v[c[0]:c[0] + 100] *= 2.0 ** 20              # key tile 0 of request 0, both halves
        v[c[0] + 200:c[0] + 230] *= 2.0 ** 20        # part of key tile 1
        v[c[2]:c[3]] *= 2.0 ** -20                   # request 2: all of its rows tiny
        run.v_new = synth.f32_to_bf16(v)
        assert np.array_equal(synth.bf16_to_f32(run.v_new), v)
        run.dev["v"] = to_device(run.v_new, w.dtype)
        out = run.run().cpu().numpy()
        torch.cuda.synchronize()
        assert run.pool.check_device_status() == 0
        for b in range(w.B):
            got = out[c[b]:c[b + 1]]
            assert np.isfinite(got).all(), f"request {b}: non-finite output"
            err = _normwise(got, run.oracle_out(b))
            print(f"request {b}: worst normwise error {err:.2e}")
            assert err <= PREFILL_RTOL
    finally:
        run.close()


def test_prefill_is_batch_invariant():
    """A request's outputs do not depend on the other requests of the batch: request 0
    alone and request 0 beside two others give the same bits."""
    outs = []
    for cached, new in (([100, 0, 513], [200, 77, 140]), ([100], [200])):
        w = make_prefill("batch", cached, new, 2, 128, group=4, seed=42)
        run = PrefillRun(w)
        try:
            outs.append(run.run()[:200].cpu().numpy())
        finally:
            run.close()
    assert np.array_equal(outs[0], outs[1])


def test_prefill_full_workload_sampled_rows():
    """The benchmarked workload at full size: sampled chunk tokens against the oracle's
    decode step at their position, every output finite, sampled rows in the pages."""
    w = workloads.chunked_prefill()
    run = PrefillRun(w, poison=False)
    try:
        out = run.run()
        torch.cuda.synchronize()
        assert run.pool.check_device_status() == 0
        assert torch.isfinite(out).all()
        out = out.cpu().numpy()
        rng = np.random.default_rng(5)
        worst = 0.0
        for b in range(w.B):
            nb = int(w.new_tokens[b])
            for i in sorted({0, nb - 1, *rng.integers(0, nb, size=2).tolist()}):
                x = int(run.cu[b]) + i
                worst = max(worst, _normwise(out[x], run.oracle_row(b, i)))
                k, v = run.chunk_rows(b, i)
                assert np.array_equal(k, run.k_new[x]) and np.array_equal(v, run.v_new[x])
        print(f"prefill_bf16 sampled: worst normwise error {worst:.2e}")
        assert worst <= PREFILL_RTOL
    finally:
        run.close()


def test_prefill_then_decode_reads_the_chunk():
    """A decode step after the prefill attends over the rows the prefill wrote."""
    import oracle
    import synth
    from synth import KHIST, VHIST, Q, F32, BF16
    w = make_prefill("then_decode", [40, 0], [90, 33], 2, 128, group=2, seed=43)
    run = PrefillRun(w)
    try:
        run.run()
        # next token of every request: position t_b, leased page if needed
        B, H, HQ, D, P = w.B, w.H, w.HQ, w.D, w.P
        for b, r in enumerate(run.reqs):
            need = (int(w.seq_lens[b]) + 1 + P - 1) // P
            if need > len(r.page_table()):
                r.lease_pages(need - len(r.page_table()))
        max_pages = max(len(r.page_table()) for r in run.reqs)
        tables = np.full((B, max_pages), -1, dtype=np.int32)
        for b, r in enumerate(run.reqs):
            tables[b, :len(r.page_table())] = r.page_table()
        lens = (w.seq_lens + 1).astype(np.int32)
        q = np.stack([synth.lane_rows(w.seed, Q, 0, b, HQ, int(lens[b]) - 1, D, F32) for b in range(B)])
        k = np.stack([synth.lane_rows(w.seed, KHIST, 0, b, H, int(lens[b]) - 1, D, BF16) for b in range(B)])
        v = np.stack([synth.lane_rows(w.seed, VHIST, 0, b, H, int(lens[b]) - 1, D, BF16) for b in range(B)])
        from synth.device import to_device
        out = run.pool.paged_decode_attention(0, to_device(q), to_device(k), to_device(v),
                                              torch.from_numpy(tables).cuda(),
                                              torch.from_numpy(lens).cuda(), int(lens.max()))
        out = out.cpu().numpy()
        for b in range(B):
            t = int(lens[b])
            n = (t + P - 1) // P
            kp = synth.request_history_pages(w, KHIST, 0, b, n, t - 1)
            vp = synth.request_history_pages(w, VHIST, 0, b, n, t - 1)
            ref = oracle.paged_decode_attention(kp, vp, q[b:b + 1], k[b:b + 1], v[b:b + 1],
                                                np.arange(n, dtype=np.int32)[None, :],
                                                np.array([t], dtype=np.int32), BF16, group=2)
            assert _normwise(out[b], ref[0]) <= 5e-3
    finally:
        run.close()


def test_prefill_bad_lengths_and_pages_set_error_bits():
    w = make_prefill("bad", [5, 20], [10, 10], 1, 64, seed=44)
    run = PrefillRun(w)
    try:
        lens = run.dev["lens"].clone()
        lens[0] = 3                                   # shorter than its chunk
        run.pool.paged_prefill(0, run.dev["q"], run.dev["k"], run.dev["v"], run.dev["cu"],
                               run.dev["tables"], lens, out=run.out)
        with pytest.raises(pkv.PkvError):
            run.pool.check_device_status()
        assert run.pool.check_device_status() == 0   # cleared
        tables = run.dev["tables"].clone()
        tables[1, 0] = w.pool_pages + 5               # page id past the pool
        run.pool.paged_prefill(0, run.dev["q"], run.dev["k"], run.dev["v"], run.dev["cu"],
                               tables, run.dev["lens"], out=run.out)
        torch.cuda.synchronize()
        bits = 0
        try:
            run.pool.check_device_status()
        except pkv.PkvError as e:
            bits = str(e)
        assert "0x2" in str(bits)
        # request 0 unaffected by request 1's bad page
        got = run.out[run.cu[0]:run.cu[1]].cpu().numpy()
        assert _normwise(got, run.oracle_out(0)) <= PREFILL_RTOL
    finally:
        run.close()


# ------------------------------------------------------ request chunks --

def _chunk_inputs(seed, layer, HQ, H, D, pos, n, req=0):
    """Chunk rows pos .. pos+n-1 of one request's streams: q [n,HQ,D], k, v [n,H,D] (bf16 bits)."""
    import synth
    from synth import KHIST, VHIST, Q, BF16
    q = np.stack([synth.rows(seed, Q, layer, req, qh, pos, n, D, BF16) for qh in range(HQ)], axis=1)
    k = np.stack([synth.rows(seed, KHIST, layer, req, h, pos, n, D, BF16) for h in range(H)], axis=1)
    v = np.stack([synth.rows(seed, VHIST, layer, req, h, pos, n, D, BF16) for h in range(H)], axis=1)
    return q, k, v


def _run_chunk(req, oreq, seed, layers, HQ, H, D, n, rid=0, only_layers=None):
    import synth
    from synth.device import to_device
    pos = req.begin_chunk(n)
    assert pos == oreq.begin_chunk(n)
    outs = []
    for layer in (range(layers) if only_layers is None else only_layers):
        q, k, v = _chunk_inputs(seed, layer, HQ, H, D, pos, n, rid)
        out = req.prefill_chunk(layer, to_device(q), to_device(k), to_device(v)).cpu().numpy()
        ref = oreq.prefill_chunk(layer, synth.bf16_to_f32(q), k, v)
        assert _normwise(out, ref) <= PREFILL_RTOL
        outs.append(out)
    return outs


def _pages_equal(pool, opool, pages, layers):
    for layer in range(layers):
        kp, vp = pool.kv_pages(layer)
        for pg in pages:
            k = kp[pg].cpu().view(torch.int16).numpy().view(np.uint16)
            v = vp[pg].cpu().view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(k, opool.k[layer, pg]) and np.array_equal(v, opool.v[layer, pg])


def test_request_chunks_then_a_token_match_the_oracle_model():
    import synth
    from oracle.model import OraclePool
    from synth import KHIST, VHIST, Q, F32, BF16
    from synth.device import to_device
    layers, H, HQ, D, seed = 2, 2, 4, 128, 5
    pool = pkv.Pool(layers, 64, H, D, 16, "bf16", 1024, seed, query_heads=HQ)
    opool = OraclePool(layers, 64, H, D, 16, BF16, max_context=1024, seed=seed, query_heads=HQ)
    req, oreq = pool.request(), opool.request()
    try:
        for n in (70, 45, 1, 130):
            _run_chunk(req, oreq, seed, layers, HQ, H, D, n)
            req.commit_token()
            oreq.commit_token()
            assert req.page_table() == oreq.table and req.length == oreq.length
        c = req.counters()
        assert (c["committed_tokens"], c["cache_appends"], c["score_cells"]) == (
            oreq.committed_tokens, oreq.cache_appends, oreq.score_cells)
        # a decode token after the chunks reads their rows
        pos = req.begin_token()
        assert pos == oreq.begin_token() == 246
        for layer in range(layers):
            q = synth.lane_rows(seed, Q, layer, 0, HQ, pos, D, F32)
            k = synth.lane_rows(seed, KHIST, layer, 0, H, pos, D, BF16)
            v = synth.lane_rows(seed, VHIST, layer, 0, H, pos, D, BF16)
            out = req.append_and_attend(layer, to_device(q), to_device(k), to_device(v)).cpu().numpy()
            ref = oreq.append_and_attend(layer, q, k, v)
            assert _normwise(out, ref) <= 5e-3
        req.commit_token()
        oreq.commit_token()
        c = req.counters()
        assert (c["committed_tokens"], c["cache_appends"], c["score_cells"]) == (
            oreq.committed_tokens, oreq.cache_appends, oreq.score_cells)
        torch.cuda.synchronize()
        assert pool.check_device_status() == 0
        _pages_equal(pool, opool, req.page_table(), layers)
    finally:
        req.close()
        pool.close()


def test_chunk_abort_then_retry_matches_no_abort():
    from oracle.model import OraclePool
    from synth import BF16
    layers, H, HQ, D, seed = 2, 1, 8, 64, 9
    results = []
    for abort in (False, True):
        pool = pkv.Pool(layers, 32, H, D, 16, "bf16", 512, seed, query_heads=HQ)
        opool = OraclePool(layers, 32, H, D, 16, BF16, max_context=512, seed=seed, query_heads=HQ)
        req, oreq = pool.request(), opool.request()
        try:
            _run_chunk(req, oreq, seed, layers, HQ, H, D, 50)
            req.commit_token()
            oreq.commit_token()
            if abort:
                free0, table0 = pool.free_list(), req.page_table()
                _run_chunk(req, oreq, seed, layers, HQ, H, D, 40, only_layers=[0])
                req.abort_token()
                oreq.abort_token()
                assert pool.free_list() == free0 and req.page_table() == table0 and req.length == 50
            outs = _run_chunk(req, oreq, seed, layers, HQ, H, D, 40)
            req.commit_token()
            oreq.commit_token()
            results.append((outs, req.page_table(), pool.free_list()))
        finally:
            req.close()
            pool.close()
    (o0, t0, f0), (o1, t1, f1) = results
    assert t0 == t1 and f0 == f1
    assert all(np.array_equal(a, b) for a, b in zip(o0, o1))


def test_chunks_over_forked_pages_copy_on_write():
    from oracle.model import OraclePool
    from synth import BF16
    layers, H, HQ, D, seed = 1, 2, 4, 128, 12
    pool = pkv.Pool(layers, 40, H, D, 16, "bf16", 640, seed, query_heads=HQ)
    opool = OraclePool(layers, 40, H, D, 16, BF16, max_context=640, seed=seed, query_heads=HQ)
    parent, oparent = pool.request(), opool.request()
    child = ochild = None
    try:
        _run_chunk(parent, oparent, seed, layers, HQ, H, D, 40)          # pages 0, 1, 2 (partial)
        parent.commit_token()
        oparent.commit_token()
        child, ochild = parent.fork(), oparent.fork()
        shared = parent.page_table()
        # the child continues in the shared partial page: it gets a private copy of page 2
        _run_chunk(child, ochild, seed, layers, HQ, H, D, 30, rid=1)
        child.commit_token()
        ochild.commit_token()
        assert child.page_table()[:2] == shared[:2] and child.page_table()[2] != shared[2]
        # the parent writes page 2 in place now that only it holds it
        _run_chunk(parent, oparent, seed, layers, HQ, H, D, 20)
        parent.commit_token()
        oparent.commit_token()
        assert parent.page_table()[2] == shared[2]
        for r, o in ((parent, oparent), (child, ochild)):
            assert r.page_table() == o.table and r.length == o.length
        assert pool.free_list() == list(opool.free)
        assert [pool.page_refs(i) for i in range(40)] == opool.refs
        torch.cuda.synchronize()
        _pages_equal(pool, opool, sorted(set(parent.page_table() + child.page_table())), layers)
    finally:
        if child is not None:
            child.close()
        parent.close()
        pool.close()
