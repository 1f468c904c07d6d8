"""Host bookkeeping of the library against the oracle's pool model, bit-exact
(CPU only: bookkeeping-only pools, no device storage)."""
import numpy as np
import pytest

import paged_kv_cache_decode_gb300 as pkv
from oracle.model import OraclePool, OracleError, Status, shuffled_pages
from synth import F32, BF16, workloads
from tests.conftest import read_golden


def host_pool(layers=1, pages=64, heads=2, head_dim=4, page_size=16, dtype="f32",
              max_context=1024, seed=0):
    return pkv.Pool(layers, pages, heads, head_dim, page_size, dtype, max_context, seed,
                    host_only=True)


@pytest.mark.parametrize("pages,seed", [(1, 0), (4, 0), (4096, 1), (32768, 2), (1000, 2**63 + 5)])
def test_free_list_matches_oracle_shuffle(pages, seed):
    with host_pool(pages=pages, seed=seed, max_context=16 * pages) as p:
        assert p.free_list() == shuffled_pages(pages, seed)


def test_zero_pages_sizes_one_full_context():
    with host_pool(pages=0, max_context=100) as p:
        assert p.pages == 7


def test_pool_bytes_worked_example():
    g = read_golden("pages_counts.txt")
    with pkv.Pool(32, 512, 16, 64, 16, "bf16", 8192, host_only=True) as p:
        assert p.bytes() == g["kv_bytes_L32_H16_dh64_S8192_2byte"]


def _apply(op, req, oreq):
    """Run one operation on both sides; return the status of each."""
    name, arg = op
    st_lib = pkv.PKV_OK
    st_orc = Status.OK
    try:
        getattr(req, name)(*arg)
    except pkv.PkvError as e:
        st_lib = e.status
    try:
        getattr(oreq, name)(*arg)
    except OracleError as e:
        st_orc = e.status
    return st_lib, st_orc


def test_lease_release_begin_abort_sequences_match_oracle():
    rng = np.random.default_rng(7)
    P, pages, maxc = 16, 40, 16 * 12
    with host_pool(pages=pages, max_context=maxc, seed=9) as p:
        op_ = OraclePool(1, pages, 2, 4, P, F32, max_context=maxc, seed=9, storage=False)
        reqs = [p.request() for _ in range(4)]
        oreqs = [op_.request() for _ in range(4)]
        for step in range(3000):
            i = int(rng.integers(0, 4))
            r, o = reqs[i], oreqs[i]
            kind = int(rng.integers(0, 5))
            if kind == 0:
                op = ("lease_pages", (int(rng.integers(-1, 6)),))
            elif kind == 1:
                op = ("release_pages", ())
            elif kind == 2:
                op = ("begin_token", ())
            else:
                op = ("abort_token", ())
            a, b = _apply(op, r, o)
            assert a == b, (step, op, a, b)
            assert r.page_table() == o.table
            assert r.length == o.length
        assert p.free_list() == list(op_.free)


def test_rejected_calls_change_nothing():
    with host_pool(pages=3, max_context=32, seed=1) as p:
        r = p.request()
        snap = lambda: (r.page_table(), r.length, p.free_list())
        s0 = snap()
        for fn, st in [(r.commit_token, pkv.PKV_ERR_BAD_STATE), (r.abort_token, pkv.PKV_ERR_BAD_STATE),
                       (lambda: r.lease_pages(3), pkv.PKV_ERR_CAPACITY_EXCEEDED),
                       (lambda: r.lease_pages(-2), pkv.PKV_ERR_INVALID_ARGUMENT)]:
            with pytest.raises(pkv.PkvError) as e:
                fn()
            assert e.value.status == st and snap() == s0
        assert r.begin_token() == 0
        s1 = snap()
        for fn, st in [(r.begin_token, pkv.PKV_ERR_BAD_STATE), (r.release_pages, pkv.PKV_ERR_BAD_STATE),
                       (lambda: r.lease_pages(1), pkv.PKV_ERR_BAD_STATE),
                       (r.commit_token, pkv.PKV_ERR_BAD_STATE)]:
            with pytest.raises(pkv.PkvError) as e:
                fn()
            assert e.value.status == st and snap() == s1
        import torch
        z = torch.zeros(2, 4)
        with pytest.raises(ValueError):          # host tensors are refused by the binding
            r.append_and_attend(0, z, z, z)
        r.abort_token()
        assert snap() == s0
        # pool exhaustion
        r.lease_pages(2)
        other = p.request()
        other.lease_pages(1)
        with pytest.raises(pkv.PkvError) as e:
            p.request().lease_pages(1)
        assert e.value.status == pkv.PKV_ERR_OUT_OF_PAGES


def test_append_on_host_only_pool_reports_no_storage():
    import ctypes
    with host_pool() as p:
        r = p.request()
        r.begin_token()
        st = pkv.lib.pkv_append_and_attend(r.handle, 0, ctypes.c_void_p(16), ctypes.c_void_p(16),
                                           ctypes.c_void_p(16), ctypes.c_void_p(16), None)
        assert st == pkv.PKV_ERR_NO_STORAGE
        with pytest.raises(pkv.PkvError):
            p.kv_pages(0)
        assert st == pkv.PKV_ERR_NO_STORAGE


def test_misaligned_tensors_rejected_before_device_work():
    """q, k, v and out must start on a multiple of min(16, one head row's bytes):
    the check runs on the host before anything else touches the pointers (fake
    addresses here), and a rejected call leaves the pending token as it was."""
    import ctypes
    A = ctypes.c_void_p
    with host_pool(head_dim=64, dtype="bf16") as p:       # rows: q/out 256 B, k/v 128 B
        r = p.request()
        r.begin_token()
        aligned = [0x10000, 0x20000, 0x30000, 0x40000]
        for i, off in [(0, 4), (1, 8), (2, 2), (3, 12)]:
            ptrs = list(aligned)
            ptrs[i] += off
            st = pkv.lib.pkv_append_and_attend(r.handle, 0, *map(A, ptrs), None)
            assert st == pkv.PKV_ERR_INVALID_ARGUMENT, (i, off)
            assert b"multiple of min(16" in pkv.lib.pkv_last_error()
        st = pkv.lib.pkv_append_and_attend(r.handle, 0, *map(A, aligned), None)
        assert st == pkv.PKV_ERR_NO_STORAGE
        r.abort_token()
        assert r.length == 0
        for off_q, off_out, want in [(4, 0, pkv.PKV_ERR_INVALID_ARGUMENT),
                                     (0, 8, pkv.PKV_ERR_INVALID_ARGUMENT),
                                     (0, 0, pkv.PKV_ERR_NO_STORAGE)]:
            st = pkv.lib.pkv_paged_decode_attention(
                p.handle, 0, 2, A(0x10000 + off_q), A(0x20000), A(0x30000), A(0x40000), 4,
                A(0x50000), 20, A(0x60000 + off_out), A(0x70000), 1 << 20, None)
            assert st == want, (off_q, off_out)
    # 4-byte rows (fp32, head_dim 1 is not a pool shape; head_dim 2 -> 8-byte rows)
    with host_pool(head_dim=2, dtype="f32") as p:
        r = p.request()
        r.begin_token()
        st = pkv.lib.pkv_append_and_attend(r.handle, 0, A(0x10008), A(0x20008), A(0x30008),
                                           A(0x40008), None)
        assert st == pkv.PKV_ERR_NO_STORAGE                 # 8-byte rows need 8-byte alignment
        st = pkv.lib.pkv_append_and_attend(r.handle, 0, A(0x10004), A(0x20000), A(0x30000),
                                           A(0x40000), None)
        assert st == pkv.PKV_ERR_INVALID_ARGUMENT
        r.abort_token()


def test_pool_destroy_refused_while_requests_live():
    p = host_pool()
    r = p.request()
    st = pkv.lib.pkv_pool_destroy(p.handle)
    assert st == pkv.PKV_ERR_BAD_STATE
    r.close()
    p.close()


def test_destroy_returns_pages():
    with host_pool(pages=10, seed=4) as p:
        r = p.request()
        r.lease_pages(4)
        r.begin_token()
        r.close()
        assert p.free_pages == 10


def test_ragged_churn_tables_match_oracle():
    """The fragmented-pool recipe: 10k seeded lease/release cycles, then every request
    leases exactly its pages.  Page tables and free list are bit-identical."""
    w = workloads.ragged()
    ops = workloads.churn_ops(w)
    with pkv.Pool(1, w.pool_pages, w.H, w.D, w.P, "bf16", w.max_context, w.seed,
                  host_only=True) as p:
        op_ = OraclePool(1, w.pool_pages, w.H, w.D, w.P, BF16, max_context=w.max_context,
                         seed=w.seed, storage=False)
        reqs = [p.request() for _ in range(w.B)]
        oreqs = [op_.request() for _ in range(w.B)]
        for r_i, kind, cnt in ops:
            op = ("lease_pages", (cnt,)) if kind == workloads.LEASE else ("release_pages", ())
            a, b = _apply(op, reqs[r_i], oreqs[r_i])
            assert a == b
        for b in range(w.B):
            _apply(("release_pages", ()), reqs[b], oreqs[b])
            _apply(("lease_pages", (int(w.n_pages[b]),)), reqs[b], oreqs[b])
        for r, o in zip(reqs, oreqs):
            assert r.page_table() == o.table
        assert p.free_list() == list(op_.free)
        used = sorted(x for r in reqs for x in r.page_table())
        assert len(used) == len(set(used)) == int(w.n_pages.sum())


# ------------------------------------------------------------ prefix sharing --

def _refs(pool, n):
    return [pool.page_refs(i) for i in range(n)]


def test_fork_shares_pages_and_copy_on_write_leases_a_private_page():
    P, pages = 16, 12
    with host_pool(pages=pages, max_context=16 * 8, seed=3) as p:
        op_ = OraclePool(1, pages, 2, 4, P, F32, max_context=16 * 8, seed=3, storage=False)
        r, o = p.request(), op_.request()
        r.lease_pages(3)
        o.lease_pages(3)
        # a mid-page length cannot be reached on a host-only pool, so share three pages
        c, oc = r.fork(), o.fork()
        assert c.page_table() == r.page_table() == oc.table
        assert _refs(p, pages) == op_.refs and sorted(set(op_.refs)) == [0, 2]
        # begin at position 0 of page 0, which is shared: copy-on-write
        assert c.begin_token() == oc.begin_token() == 0
        assert c.page_table() == oc.table and c.page_table()[0] != r.page_table()[0]
        assert _refs(p, pages) == op_.refs and p.free_list() == list(op_.free)
        c.abort_token()
        oc.abort_token()
        assert c.page_table() == r.page_table() == oc.table
        assert _refs(p, pages) == op_.refs and p.free_list() == list(op_.free)
        # releasing the parent keeps the pages the child still references
        r.release_pages()
        o.release_pages()
        assert p.free_pages == len(op_.free) == pages - 3
        c.release_pages()
        oc.release_pages()
        assert p.free_list() == list(op_.free) and p.free_pages == pages


def test_random_sequences_with_forks_match_oracle():
    rng = np.random.default_rng(11)
    P, pages, maxc = 16, 30, 16 * 10
    with host_pool(pages=pages, max_context=maxc, seed=5) as p:
        op_ = OraclePool(1, pages, 2, 4, P, F32, max_context=maxc, seed=5, storage=False)
        reqs, oreqs = [p.request()], [op_.request()]
        for step in range(3000):
            i = int(rng.integers(0, len(reqs)))
            r, o = reqs[i], oreqs[i]
            kind = int(rng.integers(0, 7))
            if kind == 5 and len(reqs) < 8:
                a = b = 0
                try:
                    c = r.fork()
                except pkv.PkvError as e:
                    a = e.status
                try:
                    oc = o.fork()
                except OracleError as e:
                    b = e.status
                assert a == b
                if a == 0:
                    reqs.append(c)
                    oreqs.append(oc)
                continue
            if kind == 6 and len(reqs) > 1:
                r.close()
                o.destroy()
                reqs.pop(i)
                oreqs.pop(i)
                continue
            op = [("lease_pages", (int(rng.integers(0, 4)),)), ("release_pages", ()),
                  ("begin_token", ()), ("abort_token", ()), ("begin_token", ())][kind % 5]
            a, b = _apply(op, r, o)
            assert a == b, (step, op, a, b)
            assert r.page_table() == o.table
        assert p.free_list() == list(op_.free)
        assert _refs(p, pages) == op_.refs


# ------------------------------------------------------------------ chunks --

def test_chunk_over_shared_pages_copies_each_and_abort_restores():
    P, pages = 16, 24
    with host_pool(pages=pages, max_context=16 * 10, seed=8) as p:
        op_ = OraclePool(1, pages, 2, 4, P, F32, max_context=16 * 10, seed=8, storage=False)
        r, o = p.request(), op_.request()
        r.lease_pages(4)
        o.lease_pages(4)
        c, oc = r.fork(), o.fork()
        # the child writes positions 0..40: pages 0, 1, 2 are shared -> three private copies
        assert c.begin_chunk(41) == oc.begin_chunk(41) == 0
        assert c.page_table() == oc.table
        assert sum(a != b for a, b in zip(c.page_table(), r.page_table())) == 3
        assert _refs(p, pages) == op_.refs and p.free_list() == list(op_.free)
        c.abort_token()
        oc.abort_token()
        assert c.page_table() == r.page_table() == oc.table
        assert _refs(p, pages) == op_.refs and p.free_list() == list(op_.free)
        # a chunk past the held pages leases the rest, in logical order
        assert c.begin_chunk(16 * 6) == oc.begin_chunk(16 * 6) == 0
        assert c.page_table() == oc.table and len(c.page_table()) == 6
        assert p.free_list() == list(op_.free)


def test_chunk_rejections_change_nothing():
    with host_pool(pages=5, max_context=64, seed=2) as p:
        r = p.request()
        snap = lambda: (r.page_table(), r.length, p.free_list())
        s0 = snap()
        for n, st in [(0, pkv.PKV_ERR_INVALID_ARGUMENT), (65, pkv.PKV_ERR_CAPACITY_EXCEEDED)]:
            with pytest.raises(pkv.PkvError) as e:
                r.begin_chunk(n)
            assert e.value.status == st and snap() == s0
        other = p.request()
        other.lease_pages(3)
        with pytest.raises(pkv.PkvError) as e:          # 3 pages needed, 2 free
            r.begin_chunk(40)
        assert e.value.status == pkv.PKV_ERR_OUT_OF_PAGES and r.page_table() == []
        assert r.begin_chunk(20) == 0
        for fn in (r.begin_token, lambda: r.begin_chunk(1), r.release_pages, r.fork):
            with pytest.raises(pkv.PkvError) as e:
                fn()
            assert e.value.status == pkv.PKV_ERR_BAD_STATE
        import torch
        z = torch.zeros(2, 4)
        with pytest.raises(ValueError):
            r.append_and_attend(0, z, z, z)
        r.abort_token()
        assert r.page_table() == [] and r.length == 0


def test_random_sequences_with_chunks_match_oracle():
    rng = np.random.default_rng(13)
    P, pages, maxc = 16, 40, 16 * 12
    with host_pool(pages=pages, max_context=maxc, seed=6) as p:
        op_ = OraclePool(1, pages, 2, 4, P, F32, max_context=maxc, seed=6, storage=False)
        reqs, oreqs = [p.request()], [op_.request()]
        for step in range(3000):
            i = int(rng.integers(0, len(reqs)))
            r, o = reqs[i], oreqs[i]
            kind = int(rng.integers(0, 8))
            if kind == 6 and len(reqs) < 8:
                a = b = 0
                try:
                    c = r.fork()
                except pkv.PkvError as e:
                    a = e.status
                try:
                    oc = o.fork()
                except OracleError as e:
                    b = e.status
                assert a == b
                if a == 0:
                    reqs.append(c)
                    oreqs.append(oc)
                continue
            if kind == 7 and len(reqs) > 1:
                r.close()
                o.destroy()
                reqs.pop(i)
                oreqs.pop(i)
                continue
            op = [("lease_pages", (int(rng.integers(0, 4)),)), ("release_pages", ()),
                  ("begin_token", ()), ("abort_token", ()), ("begin_chunk", (int(rng.integers(1, 70)),)),
                  ("abort_token", ()), ("begin_chunk", (int(rng.integers(1, 5)),))][kind % 7]
            a, b = _apply(op, r, o)
            assert a == b, (step, op, a, b)
            assert r.page_table() == o.table
        assert p.free_list() == list(op_.free)
        assert _refs(p, pages) == op_.refs


def test_sharer_leaving_during_a_pending_copy_on_write_frees_nothing_held():
    """The child writes into a shared page (copy-on-write) and the parent is destroyed
    while that token is pending: the shared page stays held by the child, and the
    abort puts it back in the child's table (commit, which frees it, runs on the GPU)."""
    with host_pool(pages=6, max_context=64, seed=3) as p:
        op_ = OraclePool(1, 6, 2, 4, 16, F32, max_context=64, seed=3, storage=False)
        r, o = p.request(), op_.request()
        r.lease_pages(2)
        o.lease_pages(2)
        c, oc = r.fork(), o.fork()
        shared = c.page_table()[0]
        assert c.begin_token() == oc.begin_token() == 0
        r.close()
        o.destroy()
        assert shared not in p.free_list() and p.page_refs(shared) == op_.refs[shared] == 1
        c.abort_token()
        oc.abort_token()
        assert c.page_table()[0] == oc.table[0] == shared and shared not in p.free_list()
        assert p.free_list() == list(op_.free) and _refs(p, 6) == op_.refs
