"""Move seeded synthetic inputs onto the device.

Input plumbing for the GPU tests and the benchmark: builds q / k_new / v_new of a
batched step and copies request history into pool pages through given page
tables.  Holds no attention arithmetic and does not import the product
package: callers pass torch views of the pool pages.
"""
from __future__ import annotations

import numpy as np
import torch

from . import F32, KHIST, VHIST, Q, rows, request_history_pages
from .workloads import Workload

TORCH_STORAGE = {F32: torch.float32, 1: torch.bfloat16}


def step_inputs(w: Workload, layer: int = 0):
    """Host arrays of one batched step: q [B,HQ,D] fp32 (HQ = H x group query heads),
    k_new / v_new [B,H,D] storage dtype (token t_b - 1 of each request's key / value
    sequence)."""
    B, H, D = w.B, w.H, w.D
    HQ = H * getattr(w, "group", 1)
    sd = np.float32 if w.dtype == F32 else np.uint16
    q = np.empty((B, HQ, D), np.float32)
    k = np.empty((B, H, D), sd)
    v = np.empty((B, H, D), sd)
    for b in range(B):
        t = int(w.seq_lens[b])
        for qh in range(HQ):
            q[b, qh] = rows(w.seed, Q, layer, b, qh, t - 1, 1, D, F32)[0]
        for h in range(H):
            k[b, h] = rows(w.seed, KHIST, layer, b, h, t - 1, 1, D, w.dtype)[0]
            v[b, h] = rows(w.seed, VHIST, layer, b, h, t - 1, 1, D, w.dtype)[0]
    return q, k, v


def prefill_inputs(w: Workload, layer: int = 0):
    """Host arrays of one batched prefill: q [N,HQ,D] and k_new / v_new [N,H,D] in the
    storage dtype (bf16 bits or fp32; tokens t_b - n_b .. t_b - 1 of each request's
    streams, requests in order) and the row offsets cu [B+1] int32."""
    H, D, HQ = w.H, w.D, w.HQ
    n = w.new_tokens.astype(np.int64)
    cu = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    N = int(cu[-1])
    sd = np.float32 if w.dtype == F32 else np.uint16
    q = np.empty((N, HQ, D), sd)
    k = np.empty((N, H, D), sd)
    v = np.empty((N, H, D), sd)
    for b in range(w.B):
        t, nb = int(w.seq_lens[b]), int(n[b])
        if nb == 0:
            continue
        rows_ = slice(int(cu[b]), int(cu[b + 1]))
        for qh in range(HQ):
            q[rows_, qh] = rows(w.seed, Q, layer, b, qh, t - nb, nb, D, w.dtype)
        for h in range(H):
            k[rows_, h] = rows(w.seed, KHIST, layer, b, h, t - nb, nb, D, w.dtype)
            v[rows_, h] = rows(w.seed, VHIST, layer, b, h, t - nb, nb, D, w.dtype)
    return q, k, v, cu


def to_device(x: np.ndarray, dtype: int | None = None, device="cuda") -> torch.Tensor:
    """numpy -> torch on the device; uint16 arrays are bf16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x))
    if x.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(device)


def fill_history(k_pages: torch.Tensor, v_pages: torch.Tensor, w: Workload, tables: np.ndarray,
                 layer: int = 0, requests=None) -> int:
    """Write tokens 0 .. t_b - 2 of every request into its pages (slot t_b - 1 is left
    for the step's own append; with w.new_tokens, tokens 0 .. t_b - n_b - 1, the chunk
    being the prefill's).  k_pages / v_pages: [pages, H, P, D] device views of one
    layer.  Pages of a shared prefix are written once, by request 0.  Returns the
    bytes written."""
    P = w.P
    S = getattr(w, "shared_prefix", 0)
    written = 0
    reqs = range(w.B) if requests is None else requests
    for b in reqs:
        t = int(w.seq_lens[b])
        cached = t - (int(w.new_tokens[b]) if w.new_tokens is not None else 1)
        n = (t + P - 1) // P
        skip = S // P if (b != 0 and S) else 0           # request 0 owns the shared pages
        idx = torch.from_numpy(np.ascontiguousarray(tables[b, skip:n], dtype=np.int64)).to(
            k_pages.device)
        for kind, dst in ((KHIST, k_pages), (VHIST, v_pages)):
            host = request_history_pages(w, kind, layer, b, n, cached)[skip:]
            dev = to_device(np.ascontiguousarray(host), w.dtype, k_pages.device)
            dst.index_copy_(0, idx, dev)
            written += host.nbytes
    return written
