"""Pins of the fp64 oracle against facts fixed outside it (CPU only).

Each pin is chosen so that a plausible slip in the oracle fails at least one:
a wrong page / slot index or a swapped K and V fails the dense reference and
the permutation check; a missing or wrong scale, or a prefix that drops the
new key, fails the dense reference; a wrong softmax fails the closed forms.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle.model import (OraclePool, OracleError, Status, shuffled_pages, _splitmix64,
                          complete_prefix_score_cells, bytes_per_session)
from synth import F32, BF16, KHIST, VHIST, Q
from tests._helpers import PagedCase, dense_causal_last_row, to_f64
from tests.conftest import read_golden, read_golden_list

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def run_oracle(case: PagedCase, lanes=None):
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    out = oracle.paged_decode_attention(kp, vp, case.q, case.k_new, case.v_new, case.tables,
                                        case.seq_lens, case.dtype, lanes=lanes)
    return out, kp, vp


CASES = [
    # (seq_lens, H, D, P, dtype)
    ([1], 1, 1, 16, F32),
    ([5, 17, 33], 2, 2, 16, F32),
    ([16, 32, 1, 64], 3, 8, 16, F32),
    ([7, 40], 2, 4, 4, F32),
    ([23, 9, 64], 2, 8, 1, F32),
    ([31, 48, 2], 2, 8, 16, BF16),
    ([64, 15], 1, 3, 8, BF16),
]


@pytest.mark.parametrize("lens,H,D,P,dtype", CASES)
def test_matches_dense_causal_last_row(lens, H, D, P, dtype):
    """Brute force: full causal attention over the logical prefix, last row."""
    case = PagedCase(lens, H, D, P, dtype, seed=11)
    out, _, _ = run_oracle(case)
    for b, t in enumerate(case.seq_lens):
        for h in range(H):
            lane = b * H + h
            K = to_f64(case.K[lane], dtype)
            V = to_f64(case.V[lane], dtype)
            ref, cells = dense_causal_last_row(case.query_rows(b, h), K, V)
            assert cells == t * t
            np.testing.assert_allclose(out[b, h], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", [F32, BF16])
def test_contiguous_single_page_layout(dtype):
    """One page of maximum-context size per request gives the paged result."""
    lens = [37, 64, 5]
    paged = PagedCase(lens, 2, 8, 16, dtype, seed=5)
    contig = PagedCase(lens, 2, 8, 64, dtype, seed=5, n_pages=3)
    assert (contig.tables[:, 0] >= 0).all() and contig.tables.shape[1] == 1
    a, _, _ = run_oracle(paged)
    b, _, _ = run_oracle(contig)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", [F32, BF16])
def test_physical_page_permutation_invariance(dtype):
    """Relabel every physical page, move its data, rewrite the tables: same bits."""
    case = PagedCase([45, 16, 3, 70], 2, 8, 16, dtype, seed=9, n_pages=40)
    out, _, _ = run_oracle(case)
    pi = np.random.default_rng(1).permutation(case.n_pages).astype(np.int32)
    k2 = np.empty_like(case.k_pool)
    v2 = np.empty_like(case.v_pool)
    k2[pi] = case.k_pool
    v2[pi] = case.v_pool
    tables = np.where(case.tables >= 0, pi[np.maximum(case.tables, 0)], -1).astype(np.int32)
    out2 = oracle.paged_decode_attention(k2, v2, case.q, case.k_new, case.v_new, tables,
                                         case.seq_lens, dtype)
    assert np.array_equal(out, out2)


def test_single_key_returns_new_value_exactly():
    """t = 1: one softmax weight of exactly 1, so out = v_new."""
    for dtype in (F32, BF16):
        case = PagedCase([1, 1], 3, 8, 16, dtype, seed=2)
        out, _, _ = run_oracle(case)
        assert np.array_equal(out, to_f64(case.v_new, dtype))


def test_zero_query_and_equal_keys_average_values():
    """q = 0, or all keys equal: uniform weights, out = mean of the value rows."""
    case = PagedCase([50, 3], 2, 4, 16, F32, seed=3)
    case.q[:] = 0
    out, _, _ = run_oracle(case)
    for b, t in enumerate(case.seq_lens):
        for h in range(2):
            mean = to_f64(case.V[b * 2 + h], F32).mean(axis=0)
            np.testing.assert_allclose(out[b, h], mean, rtol=0, atol=1e-14)
    case = PagedCase([29], 1, 4, 16, F32, seed=4)
    case.k_pool[:] = np.float32(0.5)
    case.k_new[:] = np.float32(0.5)
    out, _, _ = run_oracle(case)
    np.testing.assert_allclose(out[0, 0], to_f64(case.V[0], F32).mean(axis=0), rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value():
    """One key aligned with q and far larger than the rest takes all the weight."""
    case = PagedCase([20], 1, 4, 16, F32, seed=6)
    j = 7
    pg, slot = case.tables[0, j // 16], j % 16
    case.k_pool[pg, 0, slot] = (case.q[0, 0] * 1e4).astype(np.float32)
    out, _, _ = run_oracle(case)
    np.testing.assert_allclose(out[0, 0], case.V[0][j].astype(np.float64), rtol=0, atol=1e-12)


def test_append_writes_exact_bytes_into_slot():
    for dtype in (F32, BF16):
        case = PagedCase([18, 1, 32], 2, 8, 16, dtype, seed=8)
        out, kp, vp = run_oracle(case)
        expect_k, expect_v = case.k_pool.copy(), case.v_pool.copy()
        for b, t in enumerate(case.seq_lens):
            pg, slot = case.tables[b, (t - 1) // 16], (t - 1) % 16
            expect_k[pg, :, slot] = case.k_new[b]
            expect_v[pg, :, slot] = case.v_new[b]
        assert kp.tobytes() == expect_k.tobytes()
        assert vp.tobytes() == expect_v.tobytes()


def test_lane_subset_matches_full_run():
    case = PagedCase([40, 9, 77], 3, 8, 16, BF16, seed=12)
    full, _, _ = run_oracle(case)
    lanes = [8, 0, 4]
    part, _, _ = run_oracle(case, lanes=lanes)
    for lane in lanes:
        b, h = divmod(lane, 3)
        assert np.array_equal(part[b, h], full[b, h])


def test_out_of_range_page_is_rejected():
    case = PagedCase([20], 1, 4, 16, F32, seed=1)
    case.tables[0, 1] = case.n_pages
    with pytest.raises(ValueError):
        run_oracle(case)


# ---------------------------------------------------------------------------
# generator and allocator model


def test_splitmix64_published_outputs():
    g = _splitmix64(0)
    assert [next(g) for _ in range(3)] == read_golden_list("splitmix64_seed0.txt")


def test_fisher_yates_is_a_permutation_and_seeded():
    a = shuffled_pages(1000, 42)
    assert sorted(a) == list(range(1000))
    assert a == shuffled_pages(1000, 42)
    assert a != shuffled_pages(1000, 43)
    # first swap: i = n-1 exchanges with next() mod n
    g = _splitmix64(42)
    j = next(g) % 1000
    b = list(range(1000))
    b[999], b[j] = b[j], b[999]
    assert a[999] == b[999]


def _serial_fixture(layers, H, D, commit_lengths, abort_at=None, seed=0, pool_pages=4):
    """Drive the oracle pool through serial begin / append x layers / commit."""
    pool = OraclePool(layers, pool_pages, H, D, 16, F32, max_context=16 * pool_pages, seed=seed)
    req = pool.request()
    outs = []
    for t in commit_lengths:
        pos = req.begin_token()
        assert pos == t - 1
        if abort_at is not None and t == abort_at:
            for layer in range(layers - 1):
                req.append_and_attend(layer, synth.lane_rows(seed, Q, layer, 0, H, pos, D),
                                      synth.lane_rows(seed + 99, KHIST, layer, 0, H, pos, D),
                                      synth.lane_rows(seed + 99, VHIST, layer, 0, H, pos, D))
            before = (req.length, list(req.table))
            req.abort_token()
            assert req.length == t - 1
            assert before[0] == req.length
            pos = req.begin_token()
        step = []
        for layer in range(layers):
            step.append(req.append_and_attend(layer, synth.lane_rows(seed, Q, layer, 0, H, pos, D),
                                              synth.lane_rows(seed, KHIST, layer, 0, H, pos, D),
                                              synth.lane_rows(seed, VHIST, layer, 0, H, pos, D)))
        req.commit_token()
        outs.append(step)
    return pool, req, outs


def test_fixture_score_cells_and_appends():
    g = read_golden("pages_counts.txt")
    # 2 layers x 2 heads, serial commits at retained lengths 1, 2, 3
    pool, req, _ = _serial_fixture(2, 2, 2, [1, 2, 3])
    assert req.score_cells == g["cached_score_cells_fixture"]
    assert req.cache_appends == g["cache_appends_fixture"]
    assert req.committed_tokens == 3
    # the complete-prefix references at lengths 2 and 3: dense t x t grids per lane
    cells = 0
    for t in (2, 3):
        for _lane in range(4):
            Kd = np.random.default_rng(t).standard_normal((t, 2))
            _, c = dense_causal_last_row(Kd, Kd, Kd)
            cells += c
    assert cells == g["complete_prefix_score_cells_fixture"]
    assert complete_prefix_score_cells(4, [2, 3]) == cells
    assert cells - req.score_cells == g["avoided_score_cells_fixture"]
    # the loaded run: 2 lanes (1 layer x 2 heads), lengths 1, 2
    pool, req, _ = _serial_fixture(1, 2, 2, [1, 2])
    assert req.score_cells == g["loaded_cached_score_cells"]
    assert complete_prefix_score_cells(2, [1, 2]) == g["loaded_complete_prefix_score_cells"]


def test_abort_then_retry_matches_run_without_abort():
    """Abort at t = 3 leaves the visible length, table and pool as before the token;
    the retried run ends byte-identical to a run that never aborted."""
    p1, r1, o1 = _serial_fixture(2, 2, 2, [1, 2, 3, 4])
    p2, r2, o2 = _serial_fixture(2, 2, 2, [1, 2, 3, 4], abort_at=3)
    assert r1.length == r2.length == 4
    assert r1.table == r2.table
    assert list(p1.free) == list(p2.free)
    assert p1.k.tobytes() == p2.k.tobytes() and p1.v.tobytes() == p2.v.tobytes()
    for a, b in zip(o1, o2):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)
    # aborted attempts do not count: 4(1+2+3+4)
    assert r2.score_cells == 40 and r2.cache_appends == 8


def test_abort_returns_page_leased_by_begin():
    pool = OraclePool(1, 8, 1, 2, 16, F32, max_context=128, seed=7)
    req = pool.request()
    free0 = list(pool.free)
    req.begin_token()
    assert req.table == [free0[0]]
    req.abort_token()
    assert req.table == [] and list(pool.free) == free0 and req.length == 0


def test_rejected_operations_change_nothing():
    pool = OraclePool(2, 2, 1, 2, 16, F32, max_context=32, seed=1)
    req = pool.request()
    q = np.zeros((1, 2), np.float32)
    k = np.ones((1, 2), np.float32)

    def snap():
        return (req.length, list(req.table), list(pool.free), req.pending is None,
                pool.k.tobytes(), req.score_cells)

    s0 = snap()
    for fn, status in [(req.commit_token, Status.BAD_STATE), (req.abort_token, Status.BAD_STATE),
                       (lambda: req.append_and_attend(0, q, k, k), Status.BAD_STATE),
                       (lambda: req.lease_pages(3), Status.CAPACITY_EXCEEDED),
                       (lambda: req.lease_pages(-1), Status.INVALID_ARGUMENT)]:
        with pytest.raises(OracleError) as e:
            fn()
        assert e.value.status == status
        assert snap() == s0
    req.begin_token()
    req.append_and_attend(0, q, k, k)
    s1 = (req.length, list(req.table), list(pool.free))
    for fn, status in [(req.commit_token, Status.BAD_STATE), (req.begin_token, Status.BAD_STATE),
                       (lambda: req.append_and_attend(0, q, k, k), Status.BAD_STATE),
                       (lambda: req.append_and_attend(2, q, k, k), Status.INVALID_ARGUMENT),
                       (req.release_pages, Status.BAD_STATE)]:
        with pytest.raises(OracleError) as e:
            fn()
        assert e.value.status == status
        assert (req.length, list(req.table), list(pool.free)) == s1
    req.append_and_attend(1, q, k, k)
    req.commit_token()
    # capacity: fill to max_context, then begin is rejected
    for _ in range(31):
        req.begin_token()
        req.append_and_attend(0, q, k, k, compute=False)
        req.append_and_attend(1, q, k, k, compute=False)
        req.commit_token()
    assert req.length == 32
    with pytest.raises(OracleError) as e:
        req.begin_token()
    assert e.value.status == Status.CAPACITY_EXCEEDED
    # pool exhaustion: a second request finds no page
    other = pool.request()
    with pytest.raises(OracleError) as e:
        other.begin_token()
    assert e.value.status == Status.OUT_OF_PAGES
    assert other.table == [] and other.pending is None


def test_release_returns_pages_in_logical_order_and_resets():
    pool = OraclePool(1, 10, 1, 2, 16, F32, max_context=160, seed=3, storage=False)
    a, b = pool.request(), pool.request()
    a.lease_pages(3)
    b.lease_pages(2)
    ta = list(a.table)
    a.release_pages()
    assert list(pool.free)[-3:] == ta and a.table == [] and a.length == 0
    assert len(pool.free) == 8


def test_pool_bytes_worked_example():
    g = read_golden("pages_counts.txt")
    # 8192 positions = 512 pages of 16; 2-byte (bf16) storage stands in for fp16
    pool = OraclePool(32, 512, 16, 64, 16, BF16, max_context=8192, storage=False)
    assert pool.bytes() == g["kv_bytes_L32_H16_dh64_S8192_2byte"]
    assert bytes_per_session(32, 16, 64, 8192, 2) == g["kv_bytes_L32_H16_dh64_S8192_2byte"]
    # pages = 0 sizes the pool for one maximum-length context
    assert OraclePool(1, 0, 1, 2, 16, F32, max_context=100, storage=False).pages == 7


def test_bf16_decode_matches_torch():
    bits = np.array([0x0000, 0x8000, 0x3f80, 0xbf80, 0x0001, 0x7f7f, 0x4049, 0xc2f7],
                    dtype=np.uint16)
    kp = np.zeros((1, 1, 16, 8), np.uint16)
    vp = np.zeros_like(kp)
    k_new = np.zeros((1, 1, 8), np.uint16)
    v_new = bits.reshape(1, 1, 8)
    out = oracle.paged_decode_attention(kp, vp, np.zeros((1, 1, 8), np.float32), k_new, v_new,
                                        np.zeros((1, 1), np.int32), np.array([1], np.int32), BF16)
    assert np.array_equal(out[0, 0], to_f64(bits, BF16))


# ---------------------------------------------------------------------------
# grouped-query attention


def gqa_case(group=2, H=2, D=8, dtype=F32, lens=(23, 5, 40), seed=14):
    """A paged case with H KV heads plus a [B, H*group, D] query, and the same pools
    with every KV head repeated group times (a multi-head layout of the same data)."""
    case = PagedCase(list(lens), H, D, 16, dtype, seed=seed)
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((case.B, H * group, D)).astype(np.float32)
    rep = lambda x, axis: np.repeat(x, group, axis=axis)       # noqa: E731
    return (case, q, group, np.ascontiguousarray(rep(case.k_pool, 1)),
            np.ascontiguousarray(rep(case.v_pool, 1)), np.ascontiguousarray(rep(case.k_new, 1)),
            np.ascontiguousarray(rep(case.v_new, 1)))


@pytest.mark.parametrize("group,dtype", [(2, F32), (4, BF16), (8, F32), (16, BF16), (32, F32)])
def test_gqa_equals_mha_on_repeated_kv_heads(group, dtype):
    case, q, g, kp_rep, vp_rep, knew_rep, vnew_rep = gqa_case(group, dtype=dtype)
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    a = oracle.paged_decode_attention(kp, vp, q, case.k_new, case.v_new, case.tables,
                                      case.seq_lens, dtype, group=g)
    b = oracle.paged_decode_attention(kp_rep, vp_rep, q, knew_rep, vnew_rep, case.tables,
                                      case.seq_lens, dtype)
    assert np.array_equal(a, b)


def test_gqa_matches_dense_causal_per_query_head():
    group, H, D = 4, 2, 8
    case, q, g, *_ = gqa_case(group, H=H, D=D)
    out = oracle.paged_decode_attention(case.k_pool.copy(), case.v_pool.copy(), q, case.k_new,
                                        case.v_new, case.tables, case.seq_lens, F32, group=group)
    for b, t in enumerate(case.seq_lens):
        for qh in range(H * group):
            lane = b * H + qh // group
            Q = np.zeros((t, D))
            Q[-1] = q[b, qh]
            ref, _ = dense_causal_last_row(Q, to_f64(case.K[lane], F32), to_f64(case.V[lane], F32))
            np.testing.assert_allclose(out[b, qh], ref, rtol=0, atol=1e-12)


def test_group_one_is_multi_head():
    case = PagedCase([30, 7], 3, 8, 16, F32, seed=15)
    a, _, _ = run_oracle(case)
    b = oracle.paged_decode_attention(case.k_pool.copy(), case.v_pool.copy(), case.q, case.k_new,
                                      case.v_new, case.tables, case.seq_lens, F32, group=1)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# sliding window


def banded_last_row(Qrows, K, V, window):
    """Dense causal attention with each row limited to its last `window` keys."""
    Qd = np.asarray(Qrows, dtype=np.float64)
    t, D = Qd.shape
    S = Qd @ K.T / np.sqrt(D)
    i, j = np.indices((t, t))
    S = np.where((j <= i) & (j > i - window), S, -np.inf)
    S = S - S.max(axis=1, keepdims=True)
    W = np.exp(S)
    W /= W.sum(axis=1, keepdims=True)
    return (W @ V)[-1]


@pytest.mark.parametrize("window", [1, 5, 16, 17, 40])
def test_window_matches_banded_dense_reference(window):
    case = PagedCase([3, 17, 50, 33], 2, 8, 16, BF16, seed=21)
    out = oracle.paged_decode_attention(case.k_pool.copy(), case.v_pool.copy(), case.q,
                                        case.k_new, case.v_new, case.tables, case.seq_lens,
                                        BF16, window=window)
    for b, t in enumerate(case.seq_lens):
        for h in range(2):
            lane = b * 2 + h
            ref = banded_last_row(case.query_rows(b, h), to_f64(case.K[lane], BF16),
                                  to_f64(case.V[lane], BF16), window)
            np.testing.assert_allclose(out[b, h], ref, rtol=0, atol=1e-12)


def test_window_one_is_the_new_value_and_wide_window_is_full():
    case = PagedCase([9, 30], 2, 4, 16, F32, seed=22)
    one = oracle.paged_decode_attention(case.k_pool.copy(), case.v_pool.copy(), case.q, case.k_new,
                                        case.v_new, case.tables, case.seq_lens, F32, window=1)
    assert np.array_equal(one, to_f64(case.v_new, F32))
    full, _, _ = run_oracle(case)
    wide = oracle.paged_decode_attention(case.k_pool.copy(), case.v_pool.copy(), case.q, case.k_new,
                                         case.v_new, case.tables, case.seq_lens, F32, window=30)
    assert np.array_equal(full, wide)


def test_window_score_cells_are_lanes_times_min_t_w():
    pool = OraclePool(2, 4, 2, 2, 16, F32, max_context=64, seed=0, window=2)
    req = pool.request()
    for pos in range(4):
        req.begin_token()
        for layer in range(2):
            req.append_and_attend(layer, synth.lane_rows(0, Q, layer, 0, 2, pos, 2),
                                  synth.lane_rows(0, KHIST, layer, 0, 2, pos, 2),
                                  synth.lane_rows(0, VHIST, layer, 0, 2, pos, 2))
        req.commit_token()
    assert req.score_cells == 4 * (1 + 2 + 2 + 2)


# ---------------------------------------------------------------------------
# batched prefill


def prefill_case(L0s, ns, H, D, group=1, dtype=BF16, seed=30, P=16):
    """Requests with L0 cached tokens (in the pool) appending n new ones."""
    lens = [l0 + n for l0, n in zip(L0s, ns)]
    case = PagedCase(lens, H, D, P, dtype, seed=seed)
    # rows L0 .. L0+n-1 of every lane become the chunk's new rows; clear them from the pool
    cu = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    N = int(cu[-1])
    sd = np.float32 if dtype == F32 else np.uint16
    k_new = np.empty((N, H, D), sd)
    v_new = np.empty((N, H, D), sd)
    q = np.empty((N, H * group, D), np.float32)
    for b, (l0, n) in enumerate(zip(L0s, ns)):
        for i in range(n):
            pos = l0 + i
            pg, slot = case.tables[b, pos // P], pos % P
            for h in range(H):
                k_new[cu[b] + i, h] = case.K[b * H + h][pos]
                v_new[cu[b] + i, h] = case.V[b * H + h][pos]
                case.k_pool[pg, h, slot] = 0
                case.v_pool[pg, h, slot] = 0
            for qh in range(H * group):
                q[cu[b] + i, qh] = synth.rows(seed, Q, 0, b, qh, pos, 1, D, F32)[0]
    return case, q, k_new, v_new, cu


PREFILL_PINS = [([0, 0], [20, 33], 1, 0), ([5, 40], [12, 1], 2, 0), ([0, 17], [48, 16], 1, 20)]


@pytest.mark.parametrize("L0s,ns,group,window", PREFILL_PINS)
def test_prefill_matches_dense_causal_rows(L0s, ns, group, window):
    check_prefill_pin(L0s, ns, group, window)


def check_prefill_pin(L0s, ns, group, window, library=None):
    """Chunk outputs are rows L0..L0+n-1 of dense causal (banded) softmax attention."""
    H, D = 2, 8
    case, q, k_new, v_new, cu = prefill_case(L0s, ns, H, D, group)
    out = oracle.paged_prefill(case.k_pool, case.v_pool, q, k_new, v_new, cu, case.tables,
                               case.seq_lens, BF16, group=group, window=window, library=library)
    for b, (l0, n) in enumerate(zip(L0s, ns)):
        t = l0 + n
        for qh in range(H * group):
            lane = b * H + qh // group
            K, V = to_f64(case.K[lane], BF16), to_f64(case.V[lane], BF16)
            Qrows = np.zeros((t, D))
            for i in range(n):
                Qrows[l0 + i] = q[cu[b] + i, qh]
            S = Qrows @ K.T / np.sqrt(D)
            ii, jj = np.indices((t, t))
            keep = jj <= ii
            if window:
                keep &= jj > ii - window
            S = np.where(keep, S, -np.inf)
            S -= S.max(axis=1, keepdims=True)
            W = np.exp(S)
            W /= W.sum(axis=1, keepdims=True)
            ref = W @ V
            np.testing.assert_allclose(out[cu[b]:cu[b + 1], qh], ref[l0:t], rtol=0, atol=1e-12)
    # every new row landed in its slot
    for b, (l0, n) in enumerate(zip(L0s, ns)):
        for i in range(n):
            pos = l0 + i
            pg, slot = case.tables[b, pos // 16], pos % 16
            assert np.array_equal(case.k_pool[pg, :, slot], k_new[cu[b] + i])
