"""Test-only helpers: build paged inputs from the shared seeded generator and
an independent dense reference (numpy / torch library routines)."""
from __future__ import annotations

import numpy as np
import torch

import synth
from synth import KHIST, VHIST, Q, F32, BF16


def to_f64(x: np.ndarray, dtype: int) -> np.ndarray:
    """Storage values -> fp64 through torch's own bf16 conversion (not the oracle's)."""
    if dtype == F32:
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


class PagedCase:
    """A batch of requests with history already in a one-layer paged pool.

    Logical key/value row j of lane (b, h) is synth row (KHIST/VHIST, layer, b, h, j).
    Rows 0..t_b-2 are placed in the pool through the page tables; row t_b-1 is the
    new token (k_new / v_new), not yet in the pool.
    """

    def __init__(self, seq_lens, H, D, P=16, dtype=F32, n_pages=None, seed=0, layer=0,
                 rng_seed=None, max_pages=None):
        self.seq_lens = np.asarray(seq_lens, dtype=np.int32)
        self.B = B = len(self.seq_lens)
        self.H, self.D, self.P, self.dtype, self.seed, self.layer = H, D, P, dtype, seed, layer
        need = (self.seq_lens.astype(np.int64) + P - 1) // P
        self.max_pages = int(max_pages if max_pages is not None else max(1, need.max()))
        total = int(need.sum())
        self.n_pages = int(n_pages if n_pages is not None else max(total + 3, 4))
        rng = np.random.default_rng(seed if rng_seed is None else rng_seed)
        perm = rng.permutation(self.n_pages)[:total].astype(np.int32)
        self.tables = np.full((B, self.max_pages), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            self.tables[b, :need[b]] = perm[off:off + need[b]]
            off += need[b]
        sd = np.float32 if dtype == F32 else np.uint16
        self.k_pool = np.zeros((self.n_pages, H, P, D), dtype=sd)
        self.v_pool = np.zeros_like(self.k_pool)
        # poison free slots so a read of an unwritten slot shows up
        if dtype == F32:
            self.k_pool[:] = np.float32(1e3)
            self.v_pool[:] = np.float32(-1e3)
        self.K = []      # logical rows [t, D] storage dtype, per lane
        self.V = []
        self.q = np.empty((B, H, D), dtype=np.float32)
        self.k_new = np.empty((B, H, D), dtype=sd)
        self.v_new = np.empty((B, H, D), dtype=sd)
        for b in range(B):
            t = int(self.seq_lens[b])
            for h in range(H):
                K = synth.rows(seed, KHIST, layer, b, h, 0, t, D, dtype)
                V = synth.rows(seed, VHIST, layer, b, h, 0, t, D, dtype)
                self.K.append(K)
                self.V.append(V)
                for j in range(t - 1):
                    pg = self.tables[b, j // P]
                    self.k_pool[pg, h, j % P] = K[j]
                    self.v_pool[pg, h, j % P] = V[j]
                self.k_new[b, h] = K[t - 1]
                self.v_new[b, h] = V[t - 1]
                self.q[b, h] = synth.rows(seed, Q, layer, b, h, t - 1, 1, D, F32)[0]

    def query_rows(self, b, h):
        """All t query rows of a lane (the last one is q), for the dense reference."""
        t = int(self.seq_lens[b])
        return synth.rows(self.seed, Q, self.layer, b, h, 0, t, self.D, F32)


def dense_causal_last_row(Qrows: np.ndarray, K: np.ndarray, V: np.ndarray):
    """Complete-prefix reference: full causal attention over t positions with numpy
    matmul, last row returned.  Also returns the score-grid size (t * t)."""
    Qd = np.asarray(Qrows, dtype=np.float64)
    t, D = Qd.shape
    S = Qd @ K.T / np.sqrt(D)
    S = np.where(np.tril(np.ones((t, t), dtype=bool)), S, -np.inf)
    S = S - S.max(axis=1, keepdims=True)
    W = np.exp(S)
    W /= W.sum(axis=1, keepdims=True)
    O = W @ V
    return O[-1], S.size
