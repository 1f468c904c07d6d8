"""Failure injection on the host (CPU only, bookkeeping-only pools): a lease armed
to fail makes its call fail with PKV_ERR_OUT_OF_PAGES and change nothing, and the
pool then goes on exactly as the oracle's pool model does without that call
("Incremental Serving", section "Request flow", step 4; "38 · Cached generation":
rejected operations leave the state unchanged)."""
import numpy as np
import pytest

import paged_kv_cache_decode_gb300 as pkv
from oracle.model import OraclePool, OracleError

P = 16


def pools(pages=24, maxc=16 * 12, seed=5):
    lib = pkv.Pool(1, pages, 2, 4, P, "f32", maxc, seed, host_only=True)
    orc = OraclePool(1, pages, 2, 4, P, 0, max_context=maxc, seed=seed, storage=False)
    return lib, orc


def state(lib, reqs):
    return ([r.page_table() for r in reqs], [r.length for r in reqs], lib.free_list(),
            [lib.page_refs(x) for x in range(lib.pages)])


def orc_state(orc, oreqs):
    return ([list(o.table) for o in oreqs], [o.length for o in oreqs], list(orc.free),
            list(orc.refs))


def test_armed_lease_fails_its_call_and_changes_nothing():
    lib, orc = pools()
    with lib:
        r, o = lib.request(), orc.request()
        r.lease_pages(2)
        o.lease_pages(2)
        lib.inject_fault(pkv.PKV_INJECT_LEASE, 4)       # leases 1-3 succeed, the 4th fails
        r.lease_pages(3)
        o.lease_pages(3)
        before = state(lib, [r])
        with pytest.raises(pkv.PkvError) as e:
            r.lease_pages(2)                             # would take leases 4 and 5
        assert e.value.status == pkv.PKV_ERR_OUT_OF_PAGES
        assert "injected" in str(e.value)
        assert state(lib, [r]) == before == orc_state(orc, [o])
        r.lease_pages(2)                                 # disarmed: the same call now succeeds
        o.lease_pages(2)
        assert state(lib, [r]) == orc_state(orc, [o])


def test_armed_lease_in_begin_token_and_chunk():
    """begin_token at a page boundary and begin_chunk (with a copy-on-write page)
    fail whole when their leases reach the armed one."""
    lib, orc = pools()
    with lib:
        a, oa = lib.request(), orc.request()
        a.lease_pages(1)
        oa.lease_pages(1)
        b, ob = a.fork(), oa.fork()                     # page 0 shared, length 0
        reqs, oreqs = [a, b], [oa, ob]
        lib.inject_fault(pkv.PKV_INJECT_LEASE, 1)
        before = state(lib, reqs)
        with pytest.raises(pkv.PkvError) as e:
            b.begin_chunk(20)                            # copy of page 0 + one new page
        assert e.value.status == pkv.PKV_ERR_OUT_OF_PAGES
        assert state(lib, reqs) == before == orc_state(orc, oreqs)
        assert b.length == 0
        b.begin_chunk(20)                                # disarmed
        ob.begin_chunk(20)
        assert state(lib, reqs) == orc_state(orc, oreqs)
        b.abort_token()
        ob.abort_token()
        assert state(lib, reqs) == orc_state(orc, oreqs) == before
        c, oc = lib.request(), orc.request()
        reqs.append(c)
        oreqs.append(oc)
        lib.inject_fault(pkv.PKV_INJECT_LEASE, 2)
        c.begin_token()                                  # lease 1: position 0 needs a page
        oc.begin_token()
        c.abort_token()
        oc.abort_token()
        before = state(lib, reqs)
        with pytest.raises(pkv.PkvError):
            c.begin_token()                              # lease 2 is the armed one
        assert state(lib, reqs) == before == orc_state(orc, oreqs)


def test_random_walk_with_armed_leases_matches_model():
    """Random lease / release / begin / abort / fork with a lease armed now and then:
    a failed call is skipped on the model side, every state agrees after every step."""
    rng = np.random.default_rng(11)
    lib, orc = pools(pages=40)
    with lib:
        reqs, oreqs = [lib.request() for _ in range(3)], [orc.request() for _ in range(3)]
        injected = 0
        for step in range(2000):
            if rng.integers(0, 10) == 0:
                lib.inject_fault(pkv.PKV_INJECT_LEASE, int(rng.integers(1, 4)))
            i = int(rng.integers(0, len(reqs)))
            r, o = reqs[i], oreqs[i]
            kind = int(rng.integers(0, 6))
            name, args = [("lease_pages", (int(rng.integers(0, 4)),)), ("release_pages", ()),
                          ("begin_token", ()), ("begin_chunk", (int(rng.integers(1, 40)),)),
                          ("abort_token", ()), ("fork", ())][kind]
            before = state(lib, reqs)
            try:
                res = getattr(r, name)(*args)
                lib_err = None
            except pkv.PkvError as e:
                lib_err = e
            if lib_err is not None and "injected" in str(lib_err):
                injected += 1
                assert state(lib, reqs) == before, step
                continue
            try:
                ores = getattr(o, name)(*args)
                orc_err = None
            except OracleError as e:
                orc_err = e
            assert (lib_err is None) == (orc_err is None), (step, name, lib_err, orc_err)
            if name == "fork" and lib_err is None:
                if len(reqs) < 6:
                    reqs.append(res)
                    oreqs.append(ores)
                else:
                    res.close()
                    ores.destroy()
            assert state(lib, reqs) == orc_state(orc, oreqs), (step, name)
        assert injected > 20
        lib.inject_fault(pkv.PKV_INJECT_NONE)
        for r in reqs:
            r.close()


def test_inject_fault_rejects_bad_arguments():
    lib, _ = pools()
    with lib:
        for kind, arg in [(pkv.PKV_INJECT_LEASE, 0), (pkv.PKV_INJECT_LAYER, 1),
                          (pkv.PKV_INJECT_LAYER, -1), (99, 0)]:
            with pytest.raises(pkv.PkvError) as e:
                lib.inject_fault(kind, arg)
            assert e.value.status == pkv.PKV_ERR_INVALID_ARGUMENT
        with pytest.raises(pkv.PkvError) as e:
            lib.inject_fault(pkv.PKV_INJECT_DEVICE_WAIT, 0, 2_000_000)
        assert e.value.status == pkv.PKV_ERR_NO_STORAGE
        lib.inject_fault(pkv.PKV_INJECT_NONE)
