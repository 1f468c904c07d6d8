"""Random sequences of request operations on the GPU against the oracle model.

Several requests share one grouped-query pool (bf16 at head width 64, whose chunks
take the tensor-core prefill; fp32, and bf16 at head width 32, whose chunks run
through decode lanes); each step applies one
seeded random operation to the library and to the oracle model alike — a
token (every layer, then commit), a token aborted after some layers, a chunk
(prefill, every layer, then commit), a chunk aborted after some layers, a fork,
a destroy, a release.  After every step the tables, lengths, page references,
free list and counters agree exactly; every output agrees within the bars
(fp32: max abs 1e-5; bf16: 5e-3 normwise, decode and prefill alike); at the end every page a live request holds has the
same K/V bytes on both sides.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_decode_gb300 as pkv
import synth
from oracle.model import OraclePool, OracleError
from synth import BF16, F32
from synth.device import to_device
from tests._gpu import FP32_ATOL

pytestmark = pytest.mark.gpu

LAYERS, H, P = 2, 2, 16
PAGES, MAXC = 48, 192


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _normwise(out, ref):
    num = np.abs(out - ref).max(axis=-1)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-6)
    return float((num / den).max())


def _rows(rng, shape, dtype):
    x = rng.standard_normal(shape).astype(np.float32)
    return x if dtype == F32 else synth.f32_to_bf16(x)


def _q32(x):
    return synth.bf16_to_f32(x) if x.dtype == np.uint16 else x


def _err(out, ref, dtype):
    return float(np.abs(out - ref).max()) if dtype == F32 else _normwise(out, ref)


def _status(fn):
    try:
        fn()
        return 0
    except (pkv.PkvError, OracleError) as e:
        return e.status


@pytest.mark.parametrize("seed,dtype,D,G", [(1, BF16, 64, 2), (2, BF16, 64, 2), (3, F32, 64, 2),
                                            (4, BF16, 32, 1)])
def test_random_request_operations_match_oracle_model(seed, dtype, D, G):
    HQ = H * G
    rng = np.random.default_rng(seed)
    pool = pkv.Pool(LAYERS, PAGES, H, D, P, "f32" if dtype == F32 else "bf16", MAXC, seed,
                    query_heads=HQ)
    opool = OraclePool(LAYERS, PAGES, H, D, P, dtype, max_context=MAXC, seed=seed, query_heads=HQ)
    lanes = dtype == F32 or D not in (64, 128)      # chunks through decode lanes
    reqs, oreqs = [pool.request()], [opool.request()]
    worst = {"decode": 0.0, "prefill": 0.0}
    try:
        for step in range(160):
            i = int(rng.integers(0, len(reqs)))
            r, o = reqs[i], oreqs[i]
            kind = int(rng.integers(0, 9))
            if kind == 0 and len(reqs) < 5:
                a, b = _status(lambda: reqs.append(r.fork())), _status(lambda: oreqs.append(o.fork()))
                assert a == b
            elif kind == 1 and len(reqs) > 1:
                r.close()
                o.destroy()
                reqs.pop(i)
                oreqs.pop(i)
            elif kind == 2:
                assert _status(r.release_pages) == _status(o.release_pages)
            elif kind in (3, 4, 5):
                # one token: all layers and commit, or some layers and abort
                a, b = _status(r.begin_token), _status(o.begin_token)
                assert a == b, (step, a, b)
                if a == 0:
                    pos = o.pending["pos"]
                    done = LAYERS if kind != 5 else int(rng.integers(0, LAYERS))
                    for layer in range(done):
                        q = rng.standard_normal((HQ, D)).astype(np.float32)
                        k, v = _rows(rng, (H, D), dtype), _rows(rng, (H, D), dtype)
                        out = r.append_and_attend(layer, to_device(q), to_device(k), to_device(v))
                        ref = o.append_and_attend(layer, q, k, v)
                        worst["decode"] = max(worst["decode"], _err(out.cpu().numpy(), ref, dtype))
                    if kind == 5:
                        r.abort_token()
                        o.abort_token()
                    else:
                        r.commit_token()
                        o.commit_token()
                    assert r.length == o.length
                    del pos
            else:
                # one chunk: all layers and commit, or some layers and abort
                n = int(rng.integers(1, 40))
                a, b = _status(lambda: r.begin_chunk(n)), _status(lambda: o.begin_chunk(n))
                assert a == b, (step, n, a, b)
                if a == 0:
                    done = LAYERS if kind != 8 else int(rng.integers(0, LAYERS))
                    for layer in range(done):
                        q = _rows(rng, (n, HQ, D), dtype)
                        k, v = _rows(rng, (n, H, D), dtype), _rows(rng, (n, H, D), dtype)
                        out = r.prefill_chunk(layer, to_device(q), to_device(k), to_device(v))
                        ref = o.prefill_chunk(layer, _q32(q), k, v)
                        worst["prefill"] = max(worst["prefill"], _err(out.cpu().numpy(), ref, dtype))
                    if kind == 8:
                        r.abort_token()
                        o.abort_token()
                    else:
                        r.commit_token()
                        o.commit_token()
            for rr, oo in zip(reqs, oreqs):
                assert rr.page_table() == oo.table and rr.length == oo.length, step
                c = rr.counters()
                assert (c["committed_tokens"], c["cache_appends"], c["score_cells"]) == (
                    oo.committed_tokens, oo.cache_appends, oo.score_cells), step
            assert pool.free_list() == list(opool.free), step
            assert [pool.page_refs(x) for x in range(PAGES)] == opool.refs, step
        torch.cuda.synchronize()
        assert pool.check_device_status() == 0
        print(f"seed {seed}: worst decode {worst['decode']:.2e}, prefill {worst['prefill']:.2e}")
        if dtype == F32:
            assert worst["decode"] <= FP32_ATOL and worst["prefill"] <= FP32_ATOL
        else:
            assert worst["decode"] <= 5e-3 and worst["prefill"] <= 5e-3
        # every page a live request holds: the visible rows agree byte for byte
        for layer in range(LAYERS):
            kp, vp = pool.kv_pages(layer)
            for oo in oreqs:
                for j in range(oo.length):
                    pg, slot = oo.table[j // P], j % P
                    if dtype == F32:
                        k, v = kp[pg, :, slot].cpu().numpy(), vp[pg, :, slot].cpu().numpy()
                    else:
                        k = kp[pg, :, slot].cpu().view(torch.int16).numpy().view(np.uint16)
                        v = vp[pg, :, slot].cpu().view(torch.int16).numpy().view(np.uint16)
                    assert np.array_equal(k, opool.k[layer, pg, :, slot])
                    assert np.array_equal(v, opool.v[layer, pg, :, slot])
    finally:
        for rr in reqs:
            rr.close()
        pool.close()
