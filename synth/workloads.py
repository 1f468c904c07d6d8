"""Seeded recipes of the paged-decode workloads (shapes, lengths, allocator churn).

Every workload is synthetic.  Values are approximately N(0, 1) (see ``synth.c``);
lengths and allocator operation sequences come from numpy's PCG64 generator
seeded per workload.  Nothing here computes attention.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import F32, BF16

LEASE = 0
RELEASE = 1


@dataclasses.dataclass
class Workload:
    name: str
    B: int                 # requests
    layers: int
    H: int
    D: int
    P: int                 # page size (tokens)
    dtype: int             # storage dtype of K/V: F32 or BF16
    pool_pages: int
    max_context: int
    seed: int
    seq_lens: np.ndarray   # [B] int32, retained length t_b including the new token
    churn_cycles: int = 0  # seeded lease/release cycles before the final tables are leased
    group: int = 1         # query heads per KV head (H is the number of KV heads)
    window: int = 0        # sliding window in positions (0: whole prefix)
    shared_prefix: int = 0  # tokens every request shares with request 0 (a prompt), pages shared
    new_tokens: np.ndarray | None = None  # prefill: [B] chunk tokens appended (the last of seq_lens)

    @property
    def HQ(self) -> int:
        return self.H * self.group

    @property
    def n_pages(self) -> np.ndarray:
        return (self.seq_lens.astype(np.int64) + self.P - 1) // self.P

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2

    def kv_bytes(self) -> int:
        """K and V bytes the step must read: every retained row of every lane."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.H * self.D * 2 * self.elem_bytes


def tiny(seed: int = 0) -> Workload:
    """1 request, 2 layers, H=2, d_h=2, pages of 16, pool of 4 pages, fp32."""
    return Workload("tiny", 1, 2, 2, 2, 16, F32, 4, 64, seed, np.array([4], dtype=np.int32))


def single(t: int = 2048, seed: int = 1) -> Workload:
    """1 request, 12 layers, H=12, d_h=64, fp32, pool of 4096 shuffled pages."""
    return Workload(f"single_t{t}", 1, 12, 12, 64, 16, F32, 4096, 2048, seed,
                    np.array([t], dtype=np.int32))


def single_gqa(t: int = 2048, seed: int = 8) -> Workload:
    """1 request, 32 layers, 8 KV heads x 4 query heads, d_h=128, bf16, pool of 4096
    shuffled pages (a grouped-query model decoding alone)."""
    return Workload(f"single_gqa_t{t}", 1, 32, 8, 128, 16, BF16, 4096, 4096, seed,
                    np.array([t], dtype=np.int32), group=4)


def batched(dtype: int = BF16, seed: int = 2, B: int = 64, t_max: int = 4096) -> Workload:
    """64 requests, 1 layer, H=32, d_h=128, t ~ U{1..4096}, pool of 32768 pages."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, t_max + 1, size=B).astype(np.int32)
    name = "batched_" + ("f32" if dtype == F32 else "bf16")
    return Workload(name, B, 1, 32, 128, 16, dtype, 32768, t_max, seed, lens)


def ragged(seed: int = 3, B: int = 256, pool_pages: int = 600_000, cycles: int = 10_000) -> Workload:
    """256 requests, H=32, d_h=128, bf16, t = clip(round(lognormal(ln 512, 1)), 1, 32768),
    600k-page pool churned by 10k seeded lease/release cycles."""
    rng = np.random.default_rng(seed)
    lens = np.clip(np.rint(rng.lognormal(np.log(512.0), 1.0, size=B)), 1, 32768).astype(np.int32)
    return Workload("ragged", B, 1, 32, 128, 16, BF16, pool_pages, 32768, seed, lens,
                    churn_cycles=cycles)


def long_context(seed: int = 4, B: int = 16, t: int = 131072) -> Workload:
    """16 requests, H=8, d_h=128, bf16, t = 131072 each (8192 full pages)."""
    pages = B * ((t + 15) // 16)
    return Workload("long", B, 1, 8, 128, 16, BF16, pages, t, seed,
                    np.full(B, t, dtype=np.int32))


def churn_ops(w: Workload, max_count: int = 64):
    """Seeded lease/release operations: (request, LEASE, count) or (request, RELEASE, 0).

    A lease that would exceed one request's maximum context or the free pages is
    rejected by the allocator and changes nothing; both sides apply the same list.
    """
    rng = np.random.default_rng(w.seed + 1_000_003)
    req = rng.integers(0, w.B, size=w.churn_cycles)
    op = rng.integers(0, 2, size=w.churn_cycles)
    cnt = rng.integers(1, max_count + 1, size=w.churn_cycles)
    return [(int(r), int(o), int(c) if o == LEASE else 0) for r, o, c in zip(req, op, cnt)]


def gqa(group: int = 8, dtype: int = BF16, seed: int = 5, B: int = 64, t_max: int = 8192) -> Workload:
    """Grouped-query decode: 64 requests, 8 KV heads x `group` query heads, d_h=128,
    t ~ U{1..8192}, pool of 32768 shuffled pages."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, t_max + 1, size=B).astype(np.int32)
    name = f"gqa{group}_" + ("f32" if dtype == F32 else "bf16")
    return Workload(name, B, 1, 8, 128, 16, dtype, 32768, t_max, seed, lens, group=group)


def sliding_window(seed: int = 6, B: int = 64, t_max: int = 32768, window: int = 4096) -> Workload:
    """Sliding-window grouped-query decode: 64 requests, t ~ U{1..32768}, window 4096,
    8 KV heads x 4 query heads, d_h=128, bf16, pool of 140000 shuffled pages."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, t_max + 1, size=B).astype(np.int32)
    return Workload("window_bf16", B, 1, 8, 128, 16, BF16, 140000, t_max, seed, lens, group=4,
                    window=window)


def shared_prompt(seed: int = 7, B: int = 64, prefix: int = 8192, suffix_max: int = 1024) -> Workload:
    """Prefix-shared decode: 64 requests forked from one 8192-token prompt, each with its
    own suffix of U{1..1024} tokens (the new token included); 8 KV heads x 4 query heads,
    d_h=128, bf16, pool of 8192 shuffled pages."""
    rng = np.random.default_rng(seed)
    lens = (prefix + rng.integers(1, suffix_max + 1, size=B)).astype(np.int32)
    return Workload("prefix_bf16", B, 1, 8, 128, 16, BF16, 8192, prefix + suffix_max, seed, lens,
                    group=4, shared_prefix=prefix)


def chunked_prefill(seed: int = 8, B: int = 8, chunk: int = 4096, cached_max: int = 4096) -> Workload:
    """Chunked prefill: 8 requests each append a chunk of 4096 tokens after U{0..4096}
    cached ones; 8 KV heads x 4 query heads, d_h=128, bf16, pool of 8192 shuffled pages."""
    rng = np.random.default_rng(seed)
    cached = rng.integers(0, cached_max + 1, size=B)
    new = np.full(B, chunk, dtype=np.int32)
    lens = (cached + new).astype(np.int32)
    return Workload("prefill_bf16", B, 1, 8, 128, 16, BF16, 8192, cached_max + chunk, seed, lens,
                    group=4, new_tokens=new)


def chunked_prefill_f32(seed: int = 9, B: int = 8, chunk: int = 1024, cached_max: int = 1024) -> Workload:
    """Chunked prefill of an fp32 pool: 8 requests each append a chunk of 1024 tokens
    after U{0..1024} cached ones; 8 KV heads, one query head each, d_h=128, fp32,
    pool of 2048 shuffled pages."""
    rng = np.random.default_rng(seed)
    cached = rng.integers(0, cached_max + 1, size=B)
    new = np.full(B, chunk, dtype=np.int32)
    lens = (cached + new).astype(np.int32)
    return Workload("prefill_f32", B, 1, 8, 128, 16, F32, 2048, cached_max + chunk, seed, lens,
                    group=1, new_tokens=new)


def attended_pairs(w: Workload) -> int:
    """(query row, key) pairs of a prefill: sum over chunk tokens of the keys each attends,
    times the query heads."""
    total = 0
    for t, n in zip(w.seq_lens.astype(np.int64), w.new_tokens.astype(np.int64)):
        pos = np.arange(t - n, t, dtype=np.int64)          # positions of the chunk tokens
        keys = pos + 1
        if w.window:
            keys = np.minimum(keys, w.window)
        total += int(keys.sum())
    return total * w.HQ


def unique_rows(w: Workload) -> int:
    """Retained (KV lane, token) rows stored once: a shared prefix counts once."""
    lens = w.seq_lens.astype(np.int64)
    if w.window:
        lens = np.minimum(lens, w.window)
    rows = int(lens.sum())
    if w.shared_prefix:
        rows -= (w.B - 1) * w.shared_prefix
    return rows


REGISTRY = {
    "tiny": tiny,
    "single_t128": lambda: single(128),
    "single_t512": lambda: single(512),
    "single_t2048": lambda: single(2048),
    "single_gqa_t2048": lambda: single_gqa(2048),
    "batched_f32": lambda: batched(F32),
    "batched_bf16": lambda: batched(BF16),
    "ragged": ragged,
    "long": long_context,
    "gqa8_bf16": lambda: gqa(8, BF16),
    "gqa4_bf16": lambda: gqa(4, BF16),
    "gqa8_f32": lambda: gqa(8, F32),
    "gqa16_bf16": lambda: gqa(16, BF16),
    "window_bf16": sliding_window,
    "prefix_bf16": shared_prompt,
    "prefill_bf16": chunked_prefill,
    "prefill_f32": chunked_prefill_f32,
}
