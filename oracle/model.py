"""ORACLE — test infrastructure only.  Python model of the paged pool, its
free list, the per-request page tables and the per-token transaction.

Sources restated here:

* "Incremental Serving", section "Request flow": ``begin_token()`` reserves the
  next logical position; every layer calls ``append_and_attend(q, k, v)`` with
  [1, H, 1, d_h] tensors; ``commit_token()`` makes the position visible; after a
  failure ``abort_token()`` leaves the visible length unchanged.
* Same page, section "Paged KV-cache layout": per layer, key and value pages
  [physical_page, head, page_offset, head_width]; a request owns a logical page
  table; one physical page id addresses the matching page in every layer; pages
  are leased lazily as a sequence grows and returned on reset or destroy; page
  size 16 by default; a block count of 0 sizes the pool for one maximum-length
  context.
* "38 · Cached generation", sections "Bind one decoder to its model-wide cache"
  and "Assemble model-wide tolerance, work, generation, reset, and exact error
  evidence": every layer advances together; work counters advance only when a
  token commits (cache appends = layers per token, cached attention-score
  values = lanes x retained length per token); reset clears length and work;
  a rejected operation leaves the state unchanged.

Readings where the sources are silent:

* free list: FIFO queue initialised to a Fisher-Yates shuffle of 0..pages-1
  driven by SplitMix64(seed), swap index ``next() mod (i + 1)`` for i from
  pages-1 down to 1; lease pops the front, release pushes the request's pages
  to the back in logical order;
* ``abort_token`` returns a page leased by its ``begin_token`` to the front of
  the free list, so the pool is exactly as before ``begin_token``;
* the new row is written into its slot by ``append_and_attend``; it is visible
  only once committed because readers stop at the visible length;
* ``begin_token`` at ``max_context`` reports capacity exhaustion.

Prefix sharing ("Incremental Serving", section "Current scope", names page
sharing between matching prompts and copy-on-write prefix management as
future work; this is the plainest reading):

* ``fork`` makes a request that shares every page of its parent (each page
  counts its references); a page returns to the free list when its last
  reference is released;
* writing a token into a page that another request also references first
  moves the writer to a private copy: ``begin_token`` leases a fresh page for
  that logical page (from the free list's front), and the page's K/V bytes are
  copied into it before the token's row is written.  The writer keeps its
  reference to the shared page while the token is pending: ``commit_token``
  drops it (the page goes to the back of the free list if that was its last
  reference), ``abort_token`` puts the shared page back in the table and
  returns the fresh one to the front.  So a sharer that leaves while the
  token is pending cannot free a page the abort would restore.

Chunks (the batched prefill of "Incremental Serving", section "Paged KV-cache
layout", taken through the same transaction): ``begin_chunk(n)`` opens n
positions at the visible length at once.  Pages for all of them are leased
now, the shared pages among those the chunk writes are replaced by private
copies first (ascending logical index), then pages for logical indices the
request does not hold yet; ``prefill_chunk`` runs once per layer; commit makes
all n visible and counts each as a committed token; abort returns the leased
pages to the free list's front, last leased first, so the pool is exactly as
before ``begin_chunk``.
"""
from __future__ import annotations

import collections

import numpy as np

from . import F32, paged_decode_attention, paged_prefill, append as _append

MASK64 = (1 << 64) - 1


class Status:
    OK = 0
    INVALID_ARGUMENT = 1
    OUT_OF_PAGES = 2
    CAPACITY_EXCEEDED = 3
    BAD_STATE = 4


class OracleError(Exception):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def _splitmix64(seed: int):
    """SplitMix64 (Steele, Lea & Flood 2014): state += golden gamma, then mix."""
    state = seed & MASK64
    while True:
        state = (state + 0x9E3779B97F4A7C15) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        yield z ^ (z >> 31)


def shuffled_pages(n: int, seed: int) -> list:
    """Fisher-Yates shuffle of 0..n-1 with SplitMix64(seed)."""
    a = list(range(n))
    g = _splitmix64(seed)
    for i in range(n - 1, 0, -1):
        j = next(g) % (i + 1)
        a[i], a[j] = a[j], a[i]
    return a


def cached_score_cells(lanes: int, retained_lengths) -> int:
    """Score values formed by cached decode: lanes x t for each retained length t
    ("38 · Cached generation", "Count attention-score cells, not total runtime")."""
    return sum(lanes * t for t in retained_lengths)


class OraclePool:
    """Per-layer K/V pools [pages, H, P, D] (storage dtype) plus a FIFO free list."""

    def __init__(self, layers: int, pages: int, heads: int, head_dim: int, page_size: int = 16,
                 dtype: int = F32, max_context: int = 0, seed: int = 0, storage: bool = True,
                 query_heads: int = 0, window: int = 0):
        """heads: KV heads stored per page; query_heads: heads of the query (0 = heads),
        a multiple of heads (grouped-query attention); window: attend to the last
        `window` positions only (0 = the whole prefix)."""
        if layers < 1 or heads < 1 or head_dim < 1 or page_size < 1 or max_context < 1 or pages < 0:
            raise OracleError(Status.INVALID_ARGUMENT, "bad pool geometry")
        query_heads = query_heads or heads
        if query_heads % heads:
            raise OracleError(Status.INVALID_ARGUMENT, "query heads not a multiple of KV heads")
        self.HQ, self.group = query_heads, query_heads // heads
        self.window = window
        if pages == 0:
            pages = -(-max_context // page_size)       # one maximum-length context
        self.layers, self.pages, self.H, self.D, self.P = layers, pages, heads, head_dim, page_size
        self.dtype, self.max_context = dtype, max_context
        self.max_pages_per_request = -(-max_context // page_size)
        self.free = collections.deque(shuffled_pages(pages, seed))
        self.refs = [0] * pages                       # references per physical page
        sd = np.float32 if dtype == F32 else np.uint16
        if storage:
            self.k = np.zeros((layers, pages, heads, page_size, head_dim), dtype=sd)
            self.v = np.zeros_like(self.k)
        else:
            self.k = self.v = None
        self.requests = []

    def bytes(self) -> int:
        """Device bytes of the K and V pools: 2 * layers * pages * P * H * D * element size."""
        es = 4 if self.dtype == F32 else 2
        return 2 * self.layers * self.pages * self.P * self.H * self.D * es

    def request(self) -> "OracleRequest":
        r = OracleRequest(self)
        self.requests.append(r)
        return r

    def _lease(self) -> int:
        page = self.free.popleft()
        self.refs[page] = 1
        return page

    def _drop(self, page: int, front: bool = False) -> None:
        self.refs[page] -= 1
        if self.refs[page] == 0:
            (self.free.appendleft if front else self.free.append)(page)


class OracleRequest:
    """One request: logical page table, visible length, pending token, counters."""

    def __init__(self, pool: OraclePool):
        self.pool = pool
        self.table = []
        self.length = 0
        self.pending = None             # dict(pos, leased, appended:set) while a token is open
        self.committed_tokens = 0
        self.cache_appends = 0
        self.score_cells = 0

    # -- leasing ---------------------------------------------------------------
    def lease_pages(self, n: int) -> None:
        p = self.pool
        if self.pending is not None:
            raise OracleError(Status.BAD_STATE, "token pending")
        if n < 0:
            raise OracleError(Status.INVALID_ARGUMENT, "negative count")
        if len(self.table) + n > p.max_pages_per_request:
            raise OracleError(Status.CAPACITY_EXCEEDED, "beyond one maximum-length context")
        if n > len(p.free):
            raise OracleError(Status.OUT_OF_PAGES, "pool exhausted")
        for _ in range(n):
            self.table.append(p._lease())

    def release_pages(self) -> None:
        """Reset: every page back to the pool (logical order), length and work zeroed."""
        if self.pending is not None:
            raise OracleError(Status.BAD_STATE, "token pending")
        for page in self.table:
            self.pool._drop(page)
        self.table = []
        self.length = 0
        self.committed_tokens = self.cache_appends = self.score_cells = 0

    def destroy(self) -> None:
        if self.pending is not None:
            self.abort_token()
        self.release_pages()
        self.pool.requests.remove(self)

    def fork(self) -> "OracleRequest":
        """A new request sharing every page of this one, at the same visible length."""
        if self.pending is not None:
            raise OracleError(Status.BAD_STATE, "token pending")
        child = self.pool.request()
        child.table = list(self.table)
        child.length = self.length
        for page in self.table:
            self.pool.refs[page] += 1
        return child

    # -- the transaction ------------------------------------------------------
    def begin_token(self) -> int:
        return self._begin(1, chunk=False)

    def begin_chunk(self, n: int) -> int:
        """Open a chunk of n tokens at the visible length (batched prefill)."""
        if n < 1:
            raise OracleError(Status.INVALID_ARGUMENT, "a chunk holds at least one token")
        return self._begin(n, chunk=True)

    def _begin(self, n: int, chunk: bool) -> int:
        p = self.pool
        if self.pending is not None:
            raise OracleError(Status.BAD_STATE, "token already pending")
        if self.length + n > p.max_context:
            raise OracleError(Status.CAPACITY_EXCEEDED, "maximum context reached")
        first, last = self.length // p.P, (self.length + n - 1) // p.P
        held = len(self.table)
        shared = [i for i in range(first, min(last, held - 1) + 1) if p.refs[self.table[i]] > 1]
        new = max(0, last + 1 - held)
        if len(shared) + new > len(p.free):
            raise OracleError(Status.OUT_OF_PAGES, "pool exhausted")
        cow = []
        for idx in shared:
            # the page is shared: write into a private copy
            old = self.table[idx]
            page = p._lease()
            self.table[idx] = page
            if p.k is not None:
                p.k[:, page] = p.k[:, old]
                p.v[:, page] = p.v[:, old]
            cow.append((idx, old, page))
        leased = [p._lease() for _ in range(new)]
        self.table.extend(leased)
        self.pending = dict(pos=self.length, n=n, chunk=chunk, leased=leased, cow=cow,
                            appended=set())
        return self.length

    def append_and_attend(self, layer: int, q: np.ndarray, k: np.ndarray, v: np.ndarray,
                          compute: bool = True):
        """q [HQ, D] fp32; k, v [H, D] storage dtype.  Returns out [HQ, D] fp64 (or None)."""
        p = self.pool
        if self.pending is None or self.pending["chunk"]:
            raise OracleError(Status.BAD_STATE, "no token pending")
        if not 0 <= layer < p.layers:
            raise OracleError(Status.INVALID_ARGUMENT, "layer out of range")
        if layer in self.pending["appended"]:
            raise OracleError(Status.BAD_STATE, "layer already appended for this token")
        t = self.pending["pos"] + 1
        tables = np.asarray(self.table, dtype=np.int32)[None, :]
        lens = np.asarray([t], dtype=np.int32)
        kp, vp = p.k[layer], p.v[layer]
        if compute:
            out = paged_decode_attention(kp, vp, q[None], k[None], v[None], tables, lens, p.dtype,
                                         group=p.group, window=p.window)[0]
        else:
            _append(kp, vp, k[None], v[None], tables, lens, p.dtype)
            out = None
        self.pending["appended"].add(layer)
        return out

    def prefill_chunk(self, layer: int, q: np.ndarray, k: np.ndarray, v: np.ndarray,
                      compute: bool = True):
        """One layer of the pending chunk: q [n, HQ, D] fp32; k, v [n, H, D] storage dtype.
        Returns out [n, HQ, D] fp64 (or None)."""
        p = self.pool
        if self.pending is None or not self.pending["chunk"]:
            raise OracleError(Status.BAD_STATE, "no chunk pending")
        if not 0 <= layer < p.layers:
            raise OracleError(Status.INVALID_ARGUMENT, "layer out of range")
        if layer in self.pending["appended"]:
            raise OracleError(Status.BAD_STATE, "layer already ran for this chunk")
        pos, n = self.pending["pos"], self.pending["n"]
        tables = np.asarray(self.table, dtype=np.int32)[None, :]
        kp, vp = p.k[layer], p.v[layer]
        if compute:
            out = paged_prefill(kp, vp, q, k, v, np.array([0, n], dtype=np.int32), tables,
                                np.array([pos + n], dtype=np.int32), p.dtype, group=p.group,
                                window=p.window)
        else:
            for i in range(n):
                _append(kp, vp, k[i:i + 1], v[i:i + 1], tables,
                        np.array([pos + i + 1], dtype=np.int32), p.dtype)
            out = None
        self.pending["appended"].add(layer)
        return out

    def commit_token(self) -> None:
        """Commit the pending token or chunk: every position becomes visible; the
        counters count each position as one committed token."""
        p = self.pool
        if self.pending is None:
            raise OracleError(Status.BAD_STATE, "no token pending")
        if len(self.pending["appended"]) != p.layers:
            raise OracleError(Status.BAD_STATE, "not every layer appended")
        pos, n = self.pending["pos"], self.pending["n"]
        for _, old, _ in self.pending["cow"]:
            p._drop(old)
        self.length = pos + n
        self.committed_tokens += n
        self.cache_appends += p.layers * n
        for t in range(pos + 1, pos + n + 1):
            self.score_cells += p.layers * p.HQ * (min(t, p.window) if p.window else t)
        self.pending = None

    def abort_token(self) -> None:
        if self.pending is None:
            raise OracleError(Status.BAD_STATE, "no token pending")
        p = self.pool
        for page in reversed(self.pending["leased"]):
            assert self.table.pop() == page
            p._drop(page, front=True)
        for idx, old, new in reversed(self.pending["cow"]):
            self.table[idx] = old
            p._drop(new, front=True)
        self.pending = None


def complete_prefix_score_cells(lanes: int, lengths) -> int:
    """Dense causal score grid cells rebuilt by complete-prefix replay: lanes x t^2 each."""
    return sum(lanes * t * t for t in lengths)


def bytes_per_session(layers: int, heads: int, head_dim: int, positions: int, elem_bytes: int) -> int:
    """KV-cache bytes of one session: 2 * L * H * d_h * S * element size."""
    return 2 * layers * heads * head_dim * positions * elem_bytes


__all__ = ["Status", "OracleError", "OraclePool", "OracleRequest", "shuffled_pages",
           "cached_score_cells", "complete_prefix_score_cells", "bytes_per_session"]
