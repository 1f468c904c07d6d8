"""Batched prefill through decode lanes vs the fp64 oracle, through the C ABI.

Pools the tensor-core prefill does not serve (fp32 storage; bf16 head widths other
than 64 and 128) prefill by storing every chunk row in its page and running chunk
token i of request b as one decode request of retained length L0_b + i + 1 over
request b's pages -- the n_b successive decode steps the prefill stands for.  fp32
pools of head width 64 or 128 with 1, 2 or 4 query heads per KV head and no window
run block lanes: 8 / G consecutive chunk tokens share one decode lane of the
tensor-core kernel, each lane row masked at its own token's position.  The
bars are therefore the decode ones: max abs error <= 1e-5 for fp32 storage,
normwise relative error <= 5e-3 per (token, query head) row for bf16; the K/V rows
written into the pages bit-exact.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_decode_gb300 as pkv
import synth
from oracle.model import OraclePool
from synth import BF16, F32, KHIST, Q, VHIST
from synth.device import to_device
from tests._gpu import PrefillRun, check_close, make_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


CASES = {
    # name: (cached, new, H, D, group, P, window, dtype)
    "f32_d64_mha": ([0, 37, 300], [1, 50, 200], 2, 64, 1, 16, 0, F32),
    "f32_d128_gqa4_window": ([50, 400], [300, 16], 2, 128, 4, 16, 100, F32),
    "f32_d128_mqa16_page32": ([17, 0], [90, 33], 1, 128, 16, 32, 0, F32),
    "f32_d16_window_ragged": ([0, 3, 700], [129, 255, 1], 2, 16, 1, 16, 33, F32),
    "f32_empty_requests": ([10, 5, 0], [0, 20, 0], 2, 64, 2, 16, 0, F32),
    # block lanes (fp32, head width 64 / 128, 1, 2 or 4 query heads per KV head, no
    # window): 8 / G consecutive chunk tokens share one lane of the tensor-core kernel
    "f32_d128_mha_blocks": ([0, 16, 255], [1, 17, 300], 1, 128, 1, 16, 0, F32),
    "f32_d128_gqa2_blocks": ([0, 100, 1000], [37, 8, 129], 2, 128, 2, 16, 0, F32),
    "f32_d64_gqa4_blocks_page32": ([5, 0], [3, 77], 2, 64, 4, 32, 0, F32),
    "bf16_d32_mha": ([0, 129, 40], [100, 33, 64], 2, 32, 1, 16, 0, BF16),
    "bf16_d256_mha": ([20], [70], 1, 256, 1, 16, 0, BF16),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_lanes_match_oracle(name):
    cached, new, H, D, G, P, W, dt = CASES[name]
    w = make_prefill(name, cached, new, H, D, group=G, P=P, window=W, seed=43, dtype=dt)
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
            worst = max(worst, check_close(got, run.oracle_out(b), dt, f"{name} request {b}"))
            for i in range(nb):
                k, v = run.chunk_rows(b, i)
                x = int(run.cu[b]) + i
                assert np.array_equal(k, run.k_new[x]) and np.array_equal(v, run.v_new[x])
        print(f"{name}: worst error {worst:.2e}")
    finally:
        run.close()


def test_block_lanes_many_requests():
    """Over 1024 requests (the block plan's scan loops over request chunks) of
    chunks of 0 to 9 tokens: every row against the oracle."""
    rng = np.random.default_rng(46)
    B = 1100
    new = rng.integers(0, 10, size=B)
    cached = rng.integers(0, 40, size=B)
    w = make_prefill("many", cached, new, 1, 64, group=2, seed=47, dtype=F32)
    run = PrefillRun(w)
    try:
        out = run.run().cpu().numpy()
        torch.cuda.synchronize()
        assert run.pool.check_device_status() == 0
        for b in range(0, B, 7):                    # a seventh of the requests
            if int(w.new_tokens[b]) == 0:
                continue
            check_close(out[run.cu[b]:run.cu[b + 1]], run.oracle_out(b), F32, f"request {b}")
    finally:
        run.close()


def _chunk_inputs(seed, layer, HQ, H, D, pos, n):
    q = np.stack([synth.rows(seed, Q, layer, 0, qh, pos, n, D, F32) for qh in range(HQ)], axis=1)
    k = np.stack([synth.rows(seed, KHIST, layer, 0, h, pos, n, D, F32) for h in range(H)], axis=1)
    v = np.stack([synth.rows(seed, VHIST, layer, 0, h, pos, n, D, F32) for h in range(H)], axis=1)
    return q, k, v


def test_fp32_request_chunks_abort_and_a_token_match_the_oracle_model():
    """Transactional chunks on an fp32 pool (the request's prefill scratch grows with
    the chunk), one chunk aborted after a layer and retried, then a decode token:
    outputs, tables, counters and every page's bytes as the oracle model has them."""
    layers, H, HQ, D, seed = 2, 2, 4, 64, 9
    pool = pkv.Pool(layers, 64, H, D, 16, "f32", 1024, seed, query_heads=HQ)
    opool = OraclePool(layers, 64, H, D, 16, F32, max_context=1024, seed=seed, query_heads=HQ)
    req, oreq = pool.request(), opool.request()
    try:
        for n, abort_after in ((70, None), (45, 1), (1, None), (130, None)):
            if abort_after is not None:
                pos = req.begin_chunk(n)
                assert pos == oreq.begin_chunk(n)
                q, k, v = _chunk_inputs(seed + 1, 0, HQ, H, D, pos, n)   # other values
                req.prefill_chunk(0, to_device(q), to_device(k), to_device(v))
                req.abort_token()
                oreq.abort_token()
                assert req.page_table() == oreq.table and req.length == oreq.length
            pos = req.begin_chunk(n)
            assert pos == oreq.begin_chunk(n)
            for layer in range(layers):
                q, k, v = _chunk_inputs(seed, layer, HQ, H, D, pos, n)
                out = req.prefill_chunk(layer, to_device(q), to_device(k), to_device(v))
                ref = oreq.prefill_chunk(layer, q, k, v)
                check_close(out.cpu().numpy(), ref, F32, f"chunk {n} layer {layer}")
            req.commit_token()
            oreq.commit_token()
            assert req.page_table() == oreq.table and req.length == oreq.length
        pos = req.begin_token()
        assert pos == oreq.begin_token() == 246
        for layer in range(layers):
            q = synth.lane_rows(seed, Q, layer, 0, HQ, pos, D, F32)
            k = synth.lane_rows(seed, KHIST, layer, 0, H, pos, D, F32)
            v = synth.lane_rows(seed, VHIST, layer, 0, H, pos, D, F32)
            out = req.append_and_attend(layer, to_device(q), to_device(k), to_device(v))
            check_close(out.cpu().numpy(), oreq.append_and_attend(layer, q, k, v), F32, "token")
        req.commit_token()
        oreq.commit_token()
        c = req.counters()
        assert (c["committed_tokens"], c["cache_appends"], c["score_cells"]) == (
            oreq.committed_tokens, oreq.cache_appends, oreq.score_cells)
        torch.cuda.synchronize()
        assert pool.check_device_status() == 0
        for layer in range(layers):
            kp, vp = pool.kv_pages(layer)
            for pg in req.page_table():
                assert np.array_equal(kp[pg].cpu().numpy().view(np.uint32),
                                      opool.k[layer, pg].view(np.uint32))
                assert np.array_equal(vp[pg].cpu().numpy().view(np.uint32),
                                      opool.v[layer, pg].view(np.uint32))
    finally:
        req.close()
        pool.close()


def test_lanes_prefill_bad_lengths_set_the_error_bit():
    """A request whose length is shorter than its chunk: the error word reports it and
    the other requests' rows are still right."""
    w = make_prefill("bad", [30, 40], [20, 10], 2, 64, seed=44, dtype=F32)
    run = PrefillRun(w)
    try:
        lens = run.dev["lens"].clone()
        lens[0] = 5                                   # 5 < 20 new tokens
        d = run.dev
        out = run.pool.paged_prefill(0, d["q"], d["k"], d["v"], d["cu"], d["tables"], lens)
        torch.cuda.synchronize()
        bits = run.pool.device_status_bits()
        assert bits & pkv.PKV_DEVERR_SEQ_LEN
        got = out.cpu().numpy()[run.cu[1]:run.cu[2]]
        check_close(got, run.oracle_out(1), F32, "request 1")
    finally:
        run.close()
