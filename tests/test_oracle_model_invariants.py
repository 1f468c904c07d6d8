"""The oracle's page bookkeeping (oracle/model.py) pinned on its own, without the
library: random sequences of request operations on a small pool, with
properties that follow from the sources checked after every step, and planted
mistakes in copies of the model that those checks must reject (CPU only).

The properties:

* references -- a page's reference count equals the number of request tables
  that hold it, plus one for each pending copy-on-write that still keeps the
  shared original ("Incremental Serving", section "Current scope": shared
  pages, copy-on-write);
* free list -- every page with no reference is in the free list exactly once,
  no referenced page is; so free + referenced = pages;
* tables -- a request's table covers its visible (and pending) positions and
  holds no page twice;
* contents -- every visible row of every live request holds the bytes that
  were appended at that position of that request's history (a write into a
  page another request still reads would change them);
* transactions -- an abort leaves tables, lengths, references and the free
  list exactly as they were before the begin; a rejected call changes nothing
  ("Incremental Serving", section "Request flow", step 4; "38 · Cached
  generation": rejected operations leave the state unchanged);
* commit -- makes n positions visible and counts n committed tokens, layers x
  n appends and layers x query heads x min(t, window) score cells per position
  ("38 · Cached generation", "Count attention-score cells");
* release -- the request's pages whose last reference it held go to the back
  of the free list in logical order (the allocator reading of the design).
"""
from __future__ import annotations

import copy
import os
import types

import numpy as np
import pytest

import oracle
from oracle.model import OracleError, OraclePool
from synth import F32

MODEL_SRC = os.path.join(os.path.dirname(oracle.__file__), "model.py")

LAYERS, PAGES, P, H, D = 2, 24, 4, 1, 2


def load_model(text: str | None = None):
    """The model module, or a copy built from `text` inside the oracle package."""
    if text is None:
        import oracle.model as m
        return m
    mod = types.ModuleType("oracle._model_copy")
    mod.__package__ = "oracle"
    mod.__file__ = MODEL_SRC
    exec(compile(text, MODEL_SRC, "exec"), mod.__dict__)
    return mod


def snapshot(pool):
    reqs = [r for r in pool.requests]
    return (list(pool.free), list(pool.refs),
            [(id(r), list(r.table), r.length, r.pending is not None, r.committed_tokens,
              r.cache_appends, r.score_cells) for r in reqs])


def check_invariants(pool, rows):
    """Every property above except the transaction ones, which the driver checks."""
    held = [0] * pool.pages
    for r in pool.requests:
        assert len(set(r.table)) == len(r.table), "a page twice in one table"
        end = r.length + (r.pending["n"] if r.pending else 0)
        assert len(r.table) * pool.P >= end, "table does not cover the open positions"
        for pg in r.table:
            held[pg] += 1
        if r.pending:
            for _, old, _ in r.pending["cow"]:
                held[old] += 1
    assert list(pool.refs) == held, "reference counts differ from the tables holding the pages"
    free = list(pool.free)
    assert len(set(free)) == len(free), "a page twice in the free list"
    assert sorted(free) == [pg for pg in range(pool.pages) if held[pg] == 0], \
        "free list is not exactly the unreferenced pages"
    assert len(free) + sum(1 for x in held if x) == pool.pages
    for r in pool.requests:
        want = rows[id(r)]
        assert len(want) == r.length
        for j, vals in enumerate(want):
            pg, slot = r.table[j // pool.P], j % pool.P
            for layer in range(pool.layers):
                got = pool.k[layer, pg, :, slot, :]
                assert np.array_equal(got, vals[layer]), f"row {j} of a request changed"
                assert np.array_equal(pool.v[layer, pg, :, slot, :], -vals[layer])


class Driver:
    """Seeded random operations on one pool of model module `m`."""

    def __init__(self, m, seed, window=0):
        self.m = m
        self.rng = np.random.default_rng(seed)
        self.pool = m.OraclePool(LAYERS, PAGES, H, D, P, F32, max_context=PAGES * P // 2,
                                 seed=seed, query_heads=2 * H, window=window)
        self.rows = {}          # id(request) -> visible rows: [layer][H, D] per position
        self.pend = {}          # id(request) -> (snapshot before begin, rows being written)
        self.stamp = 1.0
        self.cnt = {}           # id(request) -> counters expected
        self.quiet = {}         # id(request) -> nothing but its own appends since its begin

    # ---- helpers --------------------------------------------------------------
    def live(self):
        return list(self.pool.requests)

    def new_rows(self, n):
        out = []
        for _ in range(n):
            out.append([np.full((H, D), self.stamp + 0.25 * layer, dtype=np.float32)
                        + np.arange(D, dtype=np.float32) / 8 for layer in range(LAYERS)])
            self.stamp += 1.0
        return out

    def rejected(self, call):
        """A call that may be refused: a refusal must leave the state unchanged."""
        before = snapshot(self.pool)
        kv = (self.pool.k.copy(), self.pool.v.copy())
        try:
            call()
            return True
        except self.m.OracleError:
            assert snapshot(self.pool) == before, "a rejected call changed the state"
            assert np.array_equal(kv[0], self.pool.k) and np.array_equal(kv[1], self.pool.v)
            return False

    # ---- operations -------------------------------------------------------------
    def create(self):
        r = self.pool.request()
        self.rows[id(r)] = []
        self.cnt[id(r)] = [0, 0, 0]

    def begin(self, r, n):
        before = snapshot(self.pool)
        call = (lambda: r.begin_token()) if n == 0 else (lambda: r.begin_chunk(n))
        if self.rejected(call):
            n = max(n, 1)
            self.pend[id(r)] = (before, self.new_rows(n), set())
            self.quiet[id(r)] = True
            assert r.pending["pos"] == r.length

    def append(self, r, layer):
        before, new, done = self.pend[id(r)]
        n = len(new)
        k = np.stack([x[layer] for x in new])           # [n, H, D]
        q = np.zeros((n, self.pool.HQ, D), dtype=np.float32)
        if r.pending["chunk"]:
            ok = self.rejected(lambda: r.prefill_chunk(layer, q, k, -k, compute=False))
        else:
            ok = self.rejected(lambda: r.append_and_attend(layer, q[0], k[0], -k[0],
                                                           compute=False))
        if ok:
            done.add(layer)

    def commit(self, r):
        before, new, done = self.pend[id(r)]
        pos = r.length
        if self.rejected(r.commit_token):
            assert done == set(range(LAYERS))
            n = len(new)
            assert r.length == pos + n
            self.rows[id(r)].extend(new)
            c = self.cnt[id(r)]
            c[0] += n
            c[1] += LAYERS * n
            w = self.pool.window
            c[2] += sum(LAYERS * self.pool.HQ * (min(t, w) if w else t)
                        for t in range(pos + 1, pos + n + 1))
            assert [r.committed_tokens, r.cache_appends, r.score_cells] == c
            del self.pend[id(r)]
            del self.quiet[id(r)]
        else:
            assert done != set(range(LAYERS))

    def abort(self, r):
        before, _, _ = self.pend.pop(id(r))
        quiet = self.quiet.pop(id(r))
        r.abort_token()
        now = snapshot(self.pool)
        # the request's own table and length are as before its begin whatever happened
        # to other requests meanwhile; the free list and references too when only its
        # own appends ran in between
        mine = [e for e in now[2] if e[0] == id(r)][0]
        then = [e for e in before[2] if e[0] == id(r)][0]
        assert mine[1:3] == then[1:3], "abort did not restore the table and length"
        if quiet:
            assert now[0] == before[0], "abort did not restore the free list"
            assert now[1] == before[1], "abort did not restore the references"

    def release(self, r):
        held_once = [pg for pg in r.table if self.pool.refs[pg] == 1]
        free0 = list(self.pool.free)
        if self.rejected(r.release_pages):
            assert list(self.pool.free) == free0 + held_once, \
                "release did not push the freed pages to the back in logical order"
            self.rows[id(r)] = []
            self.cnt[id(r)] = [0, 0, 0]

    def fork(self, r):
        out = []
        if self.rejected(lambda: out.append(r.fork())):
            c = out[0]
            assert c.table == r.table and c.length == r.length
            self.rows[id(c)] = copy.deepcopy(self.rows[id(r)])
            self.cnt[id(c)] = [0, 0, 0]
            assert [c.committed_tokens, c.cache_appends, c.score_cells] == [0, 0, 0]

    def destroy(self, r):
        if id(r) in self.pend:
            self.pend.pop(id(r))
            self.quiet.pop(id(r))
        r.destroy()
        del self.rows[id(r)]

    # ---- the random walk ----------------------------------------------------------
    def run(self, steps):
        for _ in range(steps):
            live = self.live()
            op = self.rng.integers(0, 100)
            appended = None
            if not live or (op < 8 and len(live) < 5):
                self.create()
            else:
                r = live[self.rng.integers(len(live))]
                pending = id(r) in self.pend
                if pending:
                    done = self.pend[id(r)][2]
                    if op < 60 and len(done) < LAYERS:
                        self.append(r, int(self.rng.integers(LAYERS)))
                        appended = id(r)
                    elif op < 80:
                        self.commit(r)
                    elif op < 95:
                        self.abort(r)
                    else:
                        self.destroy(r)
                else:
                    if op < 55:
                        n = 0 if self.rng.integers(2) else int(self.rng.integers(1, 7))
                        self.begin(r, n)
                        appended = id(r)
                    elif op < 65:
                        self.rejected(lambda: r.lease_pages(int(self.rng.integers(0, 4))))
                    elif op < 75:
                        self.release(r)
                    elif op < 90:
                        self.fork(r)
                    else:
                        self.destroy(r)
            for k in self.quiet:
                if k != appended:
                    self.quiet[k] = False
            check_invariants(self.pool, self.rows)


def run_walks(m, seeds=range(6), steps=1500):
    for seed in seeds:
        Driver(m, seed, window=[0, 5][seed % 2]).run(steps)


def test_model_invariants_hold_on_random_walks():
    run_walks(load_model())


def test_abort_restores_the_pool_exactly():
    """Begin (with copy-on-write of a shared page and a fresh page), some layers,
    abort: the pool is byte for byte and list for list as before."""
    pool = OraclePool(LAYERS, 8, H, D, P, F32, max_context=16, seed=3, query_heads=H)
    a = pool.request()
    a.lease_pages(1)
    for i in range(3):                       # length 3, then fork: the page is shared
        a.begin_token()
        for layer in range(LAYERS):
            a.append_and_attend(layer, np.zeros((H, D), np.float32),
                                np.full((H, D), i, np.float32), np.full((H, D), -i, np.float32),
                                compute=False)
        a.commit_token()
    b = a.fork()
    rows = {id(a): [], id(b): []}
    before = snapshot(pool)
    kv = (pool.k.copy(), pool.v.copy())
    b.begin_chunk(3)                         # writes positions 3, 4, 5: the shared page, a new one
    assert b.table[0] != a.table[0] and pool.refs[a.table[0]] == 2
    b.prefill_chunk(0, np.zeros((3, H, D), np.float32), np.ones((3, H, D), np.float32),
                    np.ones((3, H, D), np.float32), compute=False)
    b.abort_token()
    assert snapshot(pool) == before
    assert np.array_equal(pool.k[:, a.table[0]], kv[0][:, a.table[0]])
    del rows


def test_commit_after_copy_on_write_drops_the_shared_page_once():
    pool = OraclePool(1, 6, H, D, P, F32, max_context=12, seed=1, query_heads=H)
    a = pool.request()
    a.lease_pages(1)
    a.begin_token()
    a.append_and_attend(0, np.zeros((H, D), np.float32), np.ones((H, D), np.float32),
                        np.ones((H, D), np.float32), compute=False)
    a.commit_token()
    b = a.fork()
    shared = a.table[0]
    assert pool.refs[shared] == 2
    b.begin_token()
    assert pool.refs[shared] == 2            # b keeps it while the token is pending
    b.append_and_attend(0, np.zeros((H, D), np.float32), np.full((H, D), 7, np.float32),
                        np.full((H, D), 7, np.float32), compute=False)
    b.commit_token()
    assert pool.refs[shared] == 1 and shared not in b.table
    a.destroy()                              # its last reference: back of the free list
    assert list(pool.free)[-1] == shared and pool.refs[shared] == 0


# ---- planted mistakes in copies of the model ----------------------------------------

MODEL_MUTANTS = {
    "commit_keeps_shared_page": ("        for _, old, _ in self.pending[\"cow\"]:\n            p._drop(old)\n",
                                 "        for _, old, _ in self.pending[\"cow\"]:\n            pass\n"),
    "abort_returns_pages_to_back": ("            assert self.table.pop() == page\n            p._drop(page, front=True)",
                                    "            assert self.table.pop() == page\n            p._drop(page, front=False)"),
    "cow_skipped_for_two_sharers": ("if p.refs[self.table[i]] > 1]", "if p.refs[self.table[i]] > 2]"),
    "fork_without_reference": ("            self.pool.refs[page] += 1", "            self.pool.refs[page] += 0"),
    "abort_keeps_private_copy": ("            self.table[idx] = old\n            p._drop(new, front=True)",
                                 "            p._drop(old, front=True)"),
    "release_in_reverse": ("        for page in self.table:\n            self.pool._drop(page)",
                           "        for page in reversed(self.table):\n            self.pool._drop(page)"),
    "one_page_short_at_boundary": ("new = max(0, last + 1 - held)", "new = max(0, last - held)"),
    "cow_copies_nothing": ("                p.k[:, page] = p.k[:, old]\n", ""),
    "drop_frees_early": ("        self.refs[page] -= 1\n        if self.refs[page] == 0:",
                         "        self.refs[page] -= 1\n        if self.refs[page] <= 1:"),
}


def test_unmutated_model_copy_passes():
    run_walks(load_model(open(MODEL_SRC).read()), seeds=range(2), steps=600)


@pytest.mark.parametrize("name", sorted(MODEL_MUTANTS))
def test_invariants_reject_model_mutant(name):
    old, new = MODEL_MUTANTS[name]
    text = open(MODEL_SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    m = load_model(text.replace(old, new))
    with pytest.raises(AssertionError):
        run_walks(m)
