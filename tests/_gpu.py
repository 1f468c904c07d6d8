"""GPU-test helpers: run one batched step through the C ABI and the same step
through the oracle, on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_decode_gb300 as pkv
import synth
from oracle.model import OraclePool
from synth import F32, BF16, KHIST, VHIST
from synth.device import fill_history, step_inputs, to_device
from synth.workloads import Workload, churn_ops, LEASE

FP32_ATOL = 1e-5        # max abs error, fp32 storage
BF16_RTOL = 5e-3        # normwise per (request, head) row, bf16 storage


def dtype_name(dtype: int) -> str:
    return "f32" if dtype == F32 else "bf16"


def check_close(out: np.ndarray, ref: np.ndarray, dtype: int, what: str = "") -> float:
    """Assert the parity bar; return the error measure."""
    out = np.asarray(out, dtype=np.float64)
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    if dtype == F32:
        err = float(np.abs(out - ref).max()) if out.size else 0.0
        assert err <= FP32_ATOL, f"{what}: max abs error {err:.3e} > {FP32_ATOL}"
        return err
    num = np.abs(out - ref).max(axis=-1)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-6)
    err = float((num / den).max()) if out.size else 0.0
    assert err <= BF16_RTOL, f"{what}: normwise relative error {err:.3e} > {BF16_RTOL}"
    return err


class BatchedRun:
    """Pool + tables from the library's allocator (mirrored by the oracle model),
    history written into the pages, one batched step run on the device."""

    def __init__(self, w: Workload, layer: int = 0, max_seq_len=None, page_table_pad=0,
                 stream=None, cuda_cores=False):
        self.w = w
        self.layer = layer
        self.pool = pkv.Pool(w.layers, w.pool_pages, w.H, w.D, w.P, dtype_name(w.dtype),
                             w.max_context, w.seed, query_heads=w.HQ, cuda_cores=cuda_cores,
                             window=w.window)
        self.opool = OraclePool(w.layers, w.pool_pages, w.H, w.D, w.P, w.dtype,
                                max_context=w.max_context, seed=w.seed, storage=False,
                                query_heads=w.HQ, window=w.window)
        self.reqs = [self.pool.request() for _ in range(w.B)]
        self.oreqs = [self.opool.request() for _ in range(w.B)]
        for r_i, kind, cnt in churn_ops(w) if w.churn_cycles else []:
            for side, reqs in ((0, self.reqs), (1, self.oreqs)):
                try:
                    if kind == LEASE:
                        reqs[r_i].lease_pages(cnt)
                    else:
                        reqs[r_i].release_pages()
                except (pkv.PkvError, oracle.OracleError):
                    pass
        if w.shared_prefix:
            # every request forks from request 0's prompt pages, then leases its suffix
            sp = w.shared_prefix // w.P
            self.reqs[0].lease_pages(sp)
            self.oreqs[0].lease_pages(sp)
            for b in range(1, w.B):
                self.reqs[b].close()
                self.oreqs[b].destroy()
                self.reqs[b] = self.reqs[0].fork()
                self.oreqs[b] = self.oreqs[0].fork()
            for b in range(w.B):
                self.reqs[b].lease_pages(int(w.n_pages[b]) - sp)
                self.oreqs[b].lease_pages(int(w.n_pages[b]) - sp)
        else:
            for b in range(w.B):
                n = int(w.n_pages[b])
                self.reqs[b].release_pages()
                self.reqs[b].lease_pages(n)
                self.oreqs[b].release_pages()
                self.oreqs[b].lease_pages(n)
        self.max_pages = int(w.n_pages.max()) + page_table_pad
        self.tables = np.full((w.B, self.max_pages), -1, dtype=np.int32)
        self.otables = np.full((w.B, self.max_pages), -1, dtype=np.int32)
        for b in range(w.B):
            t = self.reqs[b].page_table()
            self.tables[b, :len(t)] = t
            self.otables[b, :len(self.oreqs[b].table)] = self.oreqs[b].table
        self.k_pages, self.v_pages = self.pool.kv_pages(layer)
        fill_history(self.k_pages, self.v_pages, w, self.tables, layer)
        self.q, self.k_new, self.v_new = step_inputs(w, layer)
        self.max_seq_len = int(max_seq_len or w.seq_lens.max())
        self.dev = dict(q=to_device(self.q), k=to_device(self.k_new), v=to_device(self.v_new),
                        tables=torch.from_numpy(self.tables).cuda(),
                        lens=torch.from_numpy(w.seq_lens.astype(np.int32)).cuda())
        self.out = torch.full((w.B, w.HQ, w.D), float("nan"), device="cuda")
        self.ws = self.pool.workspace(w.B, self.max_seq_len)
        self.stream = stream

    def run(self):
        d = self.dev
        self.pool.paged_decode_attention(self.layer, d["q"], d["k"], d["v"], d["tables"], d["lens"],
                                         self.max_seq_len, out=self.out, workspace=self.ws,
                                         stream=self.stream)
        return self.out

    def oracle_out(self, requests=None, heads=None) -> dict:
        """Oracle output of the given requests (all by default) on a compact host pool
        holding only their pages; tables are the oracle model's own."""
        w = self.w
        requests = list(range(w.B)) if requests is None else list(requests)
        heads = list(range(w.HQ)) if heads is None else list(heads)   # query heads
        npg = [int(w.n_pages[b]) for b in requests]
        compact = {}
        for b, n in zip(requests, npg):
            for pg in self.otables[b, :n]:
                compact.setdefault(int(pg), len(compact))
        sd = np.float32 if w.dtype == F32 else np.uint16
        kp = np.zeros((len(compact), w.H, w.P, w.D), dtype=sd)
        vp = np.zeros_like(kp)
        ctab = np.full((len(requests), max(npg)), -1, dtype=np.int32)
        for i, (b, n) in enumerate(zip(requests, npg)):
            ids = np.array([compact[int(pg)] for pg in self.otables[b, :n]], dtype=np.int64)
            ctab[i, :n] = ids
            t = int(w.seq_lens[b])
            kp[ids] = synth.request_history_pages(w, KHIST, self.layer, b, n, t - 1)
            vp[ids] = synth.request_history_pages(w, VHIST, self.layer, b, n, t - 1)
        lanes = [i * w.HQ + h for i in range(len(requests)) for h in heads]
        ref = oracle.paged_decode_attention(kp, vp, self.q[requests], self.k_new[requests],
                                            self.v_new[requests], ctab,
                                            w.seq_lens[requests].astype(np.int32), w.dtype,
                                            lanes=lanes, group=w.group, window=w.window)
        return {(b, h): ref[i, h] for i, b in enumerate(requests) for h in heads}

    def appended_rows(self, b: int):
        """Device bytes of slot t_b - 1 of request b (K and V, all heads)."""
        t = int(self.w.seq_lens[b])
        pg = int(self.tables[b, (t - 1) // self.w.P])
        slot = (t - 1) % self.w.P
        k = self.k_pages[pg, :, slot].cpu()
        v = self.v_pages[pg, :, slot].cpu()
        if self.w.dtype == BF16:
            k, v = k.view(torch.int16).numpy().view(np.uint16), v.view(torch.int16).numpy().view(np.uint16)
        else:
            k, v = k.numpy(), v.numpy()
        return k, v

    def close(self):
        self.pool.close()


def make_workload(name, seq_lens, H, D, P=16, dtype=F32, pool_pages=None, seed=0, layers=1,
                  max_context=None, churn=0, group=1, window=0) -> Workload:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    n = (seq_lens.astype(np.int64) + P - 1) // P
    if pool_pages is None:
        pool_pages = int(n.sum()) + 7
    if max_context is None:
        max_context = int(max(seq_lens.max(), 1))
    return Workload(name, len(seq_lens), layers, H, D, P, dtype, int(pool_pages), int(max_context),
                    seed, seq_lens, churn_cycles=churn, group=group, window=window)


class PrefillRun:
    """A pool (the workload's storage dtype) whose requests hold their cached tokens,
    and one batched prefill of the workload's chunks through the C ABI.  Slots at and after each request's
    cached length start as NaN, so a row the prefill fails to write, or a stale row
    it reads, shows up in the output."""

    def __init__(self, w: Workload, poison: bool = True):
        from synth.device import prefill_inputs
        self.w = w
        self.pool = pkv.Pool(w.layers, w.pool_pages, w.H, w.D, w.P, dtype_name(w.dtype),
                             w.max_context, w.seed, query_heads=w.HQ, window=w.window)
        self.reqs = [self.pool.request() for _ in range(w.B)]
        for r, n in zip(self.reqs, w.n_pages):
            r.lease_pages(int(n))
        self.max_pages = max(int(w.n_pages.max()), 1)
        self.tables = np.full((w.B, self.max_pages), -1, dtype=np.int32)
        for b, r in enumerate(self.reqs):
            t = r.page_table()
            self.tables[b, :len(t)] = t
        self.k_pages, self.v_pages = self.pool.kv_pages(0)
        self.cached = (w.seq_lens - w.new_tokens).astype(np.int64)
        if poison:
            self.k_pages.fill_(float("nan"))
            self.v_pages.fill_(float("nan"))
        fill_history(self.k_pages, self.v_pages, w, self.tables, 0)
        if poison:
            pg, sl = [], []
            for b in range(w.B):
                pos = np.arange(self.cached[b], int(w.n_pages[b]) * w.P)
                pg.append(self.tables[b, pos // w.P])
                sl.append(pos % w.P)
            pg = torch.from_numpy(np.concatenate(pg).astype(np.int64)).cuda()
            sl = torch.from_numpy(np.concatenate(sl).astype(np.int64)).cuda()
            self.k_pages[pg, :, sl] = float("nan")
            self.v_pages[pg, :, sl] = float("nan")
        self.q, self.k_new, self.v_new, self.cu = prefill_inputs(w, 0)
        self.N = int(self.cu[-1])
        self.dev = dict(q=to_device(self.q), k=to_device(self.k_new), v=to_device(self.v_new),
                        cu=torch.from_numpy(self.cu).cuda(),
                        tables=torch.from_numpy(self.tables).cuda(),
                        lens=torch.from_numpy(w.seq_lens.astype(np.int32)).cuda())
        self.out = torch.full((self.N, w.HQ, w.D), float("nan"), device="cuda")

    def run(self, stream=None):
        d = self.dev
        self.pool.paged_prefill(0, d["q"], d["k"], d["v"], d["cu"], d["tables"], d["lens"],
                                out=self.out, stream=stream)
        return self.out

    def _host_pages(self, b: int, n_tokens: int):
        """Request b's pages holding its tokens 0 .. n_tokens - 1 (rest zero)."""
        w = self.w
        n = max((n_tokens + w.P - 1) // w.P, 1)
        kp = synth.request_history_pages(w, KHIST, 0, b, n, n_tokens)
        vp = synth.request_history_pages(w, VHIST, 0, b, n, n_tokens)
        return kp, vp, np.arange(n, dtype=np.int32)[None, :]

    def oracle_out(self, b: int) -> np.ndarray:
        """Oracle prefill of request b alone: [n_b, HQ, D] fp64."""
        w = self.w
        nb = int(w.new_tokens[b])
        kp, vp, table = self._host_pages(b, int(self.cached[b]))
        tail = (int(w.seq_lens[b]) + w.P - 1) // w.P
        if tail > kp.shape[0]:
            pad = np.zeros((tail - kp.shape[0],) + kp.shape[1:], dtype=kp.dtype)
            kp, vp = np.concatenate([kp, pad]), np.concatenate([vp, pad])
            table = np.arange(tail, dtype=np.int32)[None, :]
        rows = slice(int(self.cu[b]), int(self.cu[b + 1]))
        cu = np.array([0, nb], dtype=np.int32)
        return oracle.paged_prefill(kp, vp, self._q32(self.q[rows]), self.k_new[rows],
                                    self.v_new[rows], cu, table,
                                    np.array([w.seq_lens[b]], dtype=np.int32), w.dtype,
                                    group=w.group, window=w.window)

    def _q32(self, q: np.ndarray) -> np.ndarray:
        return synth.bf16_to_f32(q) if q.dtype == np.uint16 else q

    def oracle_row(self, b: int, i: int) -> np.ndarray:
        """Oracle output of chunk token i of request b, as the decode step at position
        cached + i: [HQ, D] fp64."""
        w = self.w
        pos = int(self.cached[b]) + i
        kp, vp, table = self._host_pages(b, pos + 1)
        x = int(self.cu[b]) + i
        out = oracle.paged_decode_attention(kp, vp, self._q32(self.q[x:x + 1]),
                                            self.k_new[x:x + 1], self.v_new[x:x + 1], table,
                                            np.array([pos + 1], dtype=np.int32), w.dtype,
                                            group=w.group, window=w.window)
        return out[0]

    def chunk_rows(self, b: int, i: int):
        """Device K and V bytes at chunk token i of request b (all heads)."""
        pos = int(self.cached[b]) + i
        pg = int(self.tables[b, pos // self.w.P])
        slot = pos % self.w.P
        if self.w.dtype == F32:
            return self.k_pages[pg, :, slot].cpu().numpy(), self.v_pages[pg, :, slot].cpu().numpy()
        k = self.k_pages[pg, :, slot].cpu().view(torch.int16).numpy().view(np.uint16)
        v = self.v_pages[pg, :, slot].cpu().view(torch.int16).numpy().view(np.uint16)
        return k, v

    def close(self):
        for r in self.reqs:
            r.close()
        self.pool.close()


def make_prefill(name, cached, new, H, D, group=1, P=16, window=0, seed=0, pool_pages=None,
                 dtype=BF16):
    cached = np.asarray(cached, dtype=np.int64)
    new = np.asarray(new, dtype=np.int32)
    lens = (cached + new).astype(np.int32)
    n = (lens.astype(np.int64) + P - 1) // P
    if pool_pages is None:
        pool_pages = int(n.sum()) + 13
    return Workload(name, len(lens), 1, H, D, P, dtype, int(pool_pages), int(max(lens.max(), 1)),
                    seed, lens, group=group, window=window, new_tokens=new)
