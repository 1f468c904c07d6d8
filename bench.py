#!/usr/bin/env python3
"""Paged decode attention benchmark (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl pkv|reference]

A step is one pass of the whole decode path over one batch: the plan kernel
and the fused append + split attention + merge kernel, for every request of
the workload (one layer).  Inputs are synthetic and seeded; the K/V history
is resident in HBM before timing starts.  The default workload is the
long-context batch: 16 requests x 131072 tokens, H=8, d_h=128, bf16 pages of
16 tokens (8.6 GB of K/V per step, far larger than L2, so no flush is needed).

``--impl reference`` times the fp64 CPU oracle on the host cores instead (the
only other place this script runs the oracle), one bounded sample per step.
For N > 1 (torchrun), every rank runs its own replica of the workload (weak
scaling, no data-path collective); rank 0 prints.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: achieved HBM GB/s (% of 8 TB/s) and decode tokens/s"
PREFILL_METRIC = ("batched prefill attention into the paged cache: TFLOP/s (causal, algorithmic "
                  "FLOPs) and new tokens/s")
# further decode workloads measured in the default (long-context) run, each a short record
EXTRA_WORKLOADS = ("batched_bf16", "batched_f32", "ragged")
NOMINAL_HBM_GBS = 8000.0
DECODE_SRC = os.path.join(ROOT, "paged_kv_cache_decode_gb300", "csrc", "decode.cu")
PREFILL_SRC = os.path.join(ROOT, "paged_kv_cache_decode_gb300", "csrc", "prefill.cu")
SHARED_SRC = os.path.join(ROOT, "paged_kv_cache_decode_gb300", "csrc", "shared_prefix.cu")
TRAFFIC_DIR = os.path.join(ROOT, "profiles")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------- workload --

def make_workload(name: str, rank: int = 0, requests: int = 0):
    """The named workload; ``requests`` > 0 keeps only its first requests (small
    profiling captures that hold a few GB on the device).  The pool shrinks to
    match: exactly the kept pages for the long-context workload (all its pages are
    used), else at most twice them, so the tables still scatter over a pool."""
    from synth import workloads
    w = workloads.REGISTRY[name]()
    w.seed += 1000 * rank          # each replica draws its own values
    if 0 < requests < w.B:
        w.B = requests
        w.seq_lens = w.seq_lens[:requests].copy()
        if w.new_tokens is not None:
            w.new_tokens = w.new_tokens[:requests].copy()
        kept = int(w.n_pages.sum())
        w.pool_pages = min(w.pool_pages, kept if w.name == "long" else 2 * kept)
        w.name += f"_first{requests}"
    return w


def describe(w) -> str:
    st = "fp32" if w.elem_bytes == 4 else "bf16"
    if w.name == "long":
        return (f"long context: {w.B} requests x {int(w.seq_lens[0])} tokens, H={w.H}, d_h={w.D}, "
                f"{st} pages of {w.P}")
    if w.name.startswith("batched"):
        return (f"batched decode: {w.B} requests, t ~ U[1,4096], H={w.H}, d_h={w.D}, {st}, "
                f"pool of {w.pool_pages} shuffled pages")
    if w.name.startswith("prefix"):
        return (f"shared-prompt decode: {w.B} requests forked from one {w.shared_prefix}-token "
                f"prompt, each with its own suffix (t ~ {w.shared_prefix} + U[1,"
                f"{w.max_context - w.shared_prefix}]), {w.H} KV heads x {w.group} query heads, "
                f"d_h={w.D}, {st}")
    if w.name.startswith("window"):
        return (f"sliding-window decode: {w.B} requests, t ~ U[1,{w.max_context}], window "
                f"{w.window}, {w.H} KV heads x {w.group} query heads each, d_h={w.D}, {st}, "
                f"pool of {w.pool_pages} shuffled pages")
    if w.name.startswith("gqa"):
        return (f"grouped-query decode: {w.B} requests, t ~ U[1,{w.max_context}], {w.H} KV heads x "
                f"{w.group} query heads each, d_h={w.D}, {st}, pool of {w.pool_pages} shuffled pages")
    if w.name.startswith("prefill"):
        cached = w.seq_lens - w.new_tokens
        return (f"chunked prefill: {w.B} requests each appending {int(w.new_tokens[0])} tokens "
                f"after U[0,{int(w.max_context - w.new_tokens.max())}] cached ones (mean "
                f"{float(cached.mean()):.0f}), {w.H} KV heads x {w.group} query heads, d_h={w.D}, "
                f"{st} pages of {w.P}, causal")
    if w.name == "ragged":
        return (f"ragged fragmented pool: {w.B} requests, lognormal(ln 512, 1) lengths, H={w.H}, "
                f"d_h={w.D}, {st}, {w.pool_pages}-page pool after {w.churn_cycles} lease/release cycles")
    return w.name


def algorithmic_bytes(w) -> int:
    """Bytes one step must move: retained history K and V rows, the new rows read
    and written, q and out, page-table entries and lengths."""
    from synth.workloads import unique_rows
    es = w.elem_bytes
    # history rows read once (a window limits them; a shared prefix counts once);
    # the new row of each lane is read from k_new / v_new instead
    hist = (unique_rows(w) - w.B) * w.H * w.D * 2 * es
    new_rows = w.B * w.H * w.D * es * 2 * 2
    q_out = w.B * w.HQ * w.D * 4 * 2                             # query heads
    tables = int(w.n_pages.sum()) * 4 + w.B * 4
    return hist + new_rows + q_out + tables


def decode_config(w, world: int, shared: int = 0) -> dict:
    """The ``config`` object of a decode line; both arms print the same one."""
    alg = algorithmic_bytes(w)
    cfg = {"workload": describe(w), "name": w.name, "requests": w.B, "heads": w.H,
           "query_heads": w.HQ, "head_dim": w.D, "page_size": w.P,
           "pool_pages": w.pool_pages,
           "seq_len_max": int(w.seq_lens.max()), "tokens_retained": int(w.seq_lens.sum()),
           "storage": "bf16" if w.elem_bytes == 2 else "fp32", "accumulate": "fp32",
           "alg_bytes_per_step": alg,
           "logical_kv_bytes_per_step": logical_bytes(w),
           "l2": f"inputs larger than L2 ({alg / 1e9:.2f} GB per step, no flush)"
                 if alg > 129e6 else "inputs smaller than L2 (cache-warm)",
           "parallelism": f"replicas x{world}"}
    if shared:
        cfg["path"] = (f"shared-prefix call: the {shared}-token prompt once per KV head on the "
                       "tensor cores, each request's own positions by the split kernel, partials "
                       "merged")
    return cfg


def prefill_config(w, world: int) -> dict:
    """The ``config`` object of a prefill line; both arms print the same one."""
    kv_bytes = int(w.seq_lens.astype(np.int64).sum()) * w.H * w.D * 2 * 2
    return {"workload": describe(w), "name": w.name, "requests": w.B, "heads": w.H,
            "query_heads": w.HQ, "head_dim": w.D, "page_size": w.P,
            "pool_pages": w.pool_pages, "new_tokens": int(w.new_tokens.sum()),
            "cached_tokens": int((w.seq_lens - w.new_tokens).sum()),
            "storage": "bf16" if w.elem_bytes == 2 else "fp32", "accumulate": "fp32",
            "flops_per_step": prefill_flops(w),
            "l2": f"K/V of the step {kv_bytes / 1e9:.2f} GB, re-read across query "
                  f"tiles through L2 (no flush)",
            "parallelism": f"replicas x{world}"}


def serial_config(w, world: int) -> dict:
    """The ``config`` object of a single-request line; both arms print the same one."""
    t = int(w.seq_lens[0])
    alg = token_bytes(w, t)
    layer_alg = alg // w.layers
    heads = f"H={w.H}" if w.group == 1 else f"{w.H} KV heads x {w.group} query heads"
    st = "bf16" if w.elem_bytes == 2 else "fp32"
    return {"workload": (f"single request: {w.layers} layers, {heads}, d_h={w.D}, {st}, "
                         f"retained length t={t}, pool of {w.pool_pages} shuffled pages; "
                         "a step is one token through every layer (transactional API)"),
            "name": w.name, "layers": w.layers, "heads": w.H, "query_heads": w.HQ, "head_dim": w.D,
            "page_size": w.P, "seq_len": t, "alg_bytes_per_step": alg,
            "calls": "timed token through the C ABI (pointers taken once); e2e the same "
                     "calls, with the token's inputs of every layer copied in from pinned host "
                     "memory (one copy) and every layer's output copied back (one copy)",
            "l2": f"{layer_alg / 1e6:.1f} MB per layer, {alg / 1e6:.0f} MB per token, no flush: "
                  + ("every layer's history fits in the 129 MB L2 between tokens"
                     if alg <= 129e6 else "larger than the 129 MB L2"),
            "parallelism": f"replicas x{world}"}


def logical_bytes(w) -> int:
    """K/V bytes the attention reads counting every request's rows, shared or not."""
    lens = w.seq_lens.astype(np.int64)
    if w.window:
        lens = np.minimum(lens, w.window)
    return int((lens - 1).sum()) * w.H * w.D * 2 * w.elem_bytes


# ---------------------------------------------------------------- ranks --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def max_over_ranks(x: float, device="cpu") -> float:
    """Largest value of x over all ranks (timing only; no data-path exchange)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


# --------------------------------------------------------------- clocks --

CLOCK_FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw",
                "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
                "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, kept by timestamp."""

    def __init__(self, device_index: int = 0):
        self.proc = None
        try:
            import torch
            ident = ["-i", "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)]
        except Exception:
            ident = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(CLOCK_FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "20", *ident], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        self.samples = []

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) != len(CLOCK_FIELDS):
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                self.samples.append(dict(t=ts, sm=float(f[1]), sm_max=float(f[2]), fields=f))
            except ValueError:
                continue

    def summary(self, t0: float, t1: float) -> dict:
        win = [s for s in self.samples if t0 <= s["t"] <= t1]
        note = "samples inside the timed region"
        if not win:
            win = self.samples
            note = "no sample fell inside the timed region; all samples of the run"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in win for n, v in zip(names, s["fields"][5:9]) if v == "Active"})
        return {"sm_mhz": float(np.median([s["sm"] for s in win])),
                "sm_max_mhz": max(s["sm_max"] for s in win), "reasons": reasons,
                "samples": len(win), "note": note}


# -------------------------------------------------------------- roofline --

def measured_peak_hbm():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def measured_traffic(workload: str, kernel: str = "split_decode", source=DECODE_SRC):
    """DRAM bytes per launch of a kernel from the committed ncu summary
    profiles/traffic_<kernel>_<workload>.txt, or None when there is none or the
    kernel source changed since the counters were taken.  Several sources hash
    as the sha256 of their sha256 hex digests, in order."""
    rec = {}
    try:
        with open(os.path.join(TRAFFIC_DIR, f"traffic_{kernel}_{workload}.txt")) as f:
            for line in f:
                line = line.split("#", 1)[0].split()
                if len(line) == 2:
                    rec[line[0]] = line[1]
    except OSError:
        return None
    if isinstance(source, (list, tuple)):
        want = hashlib.sha256("".join(source_hash(x) for x in source).encode()).hexdigest()
    else:
        want = source_hash(source)
    if rec.get("source_sha256") != want or "dram_bytes_per_launch" not in rec:
        return None
    return int(rec["dram_bytes_per_launch"])


# ------------------------------------------------------------ the GPU arm --

def setup_device(w, torch, cuda_cores=False):
    """Pool, tables from the library's allocator, history in HBM, step inputs on device."""
    import paged_kv_cache_decode_gb300 as pkv
    from synth.device import fill_history, step_inputs, to_device
    from synth.workloads import churn_ops, LEASE

    pool = pkv.Pool(w.layers, w.pool_pages, w.H, w.D, w.P, "f32" if w.elem_bytes == 4 else "bf16",
                    w.max_context, w.seed, query_heads=w.HQ, cuda_cores=cuda_cores,
                    window=w.window)
    reqs = [pool.request() for _ in range(w.B)]
    for r_i, kind, cnt in (churn_ops(w) if w.churn_cycles else []):
        try:
            reqs[r_i].lease_pages(cnt) if kind == LEASE else reqs[r_i].release_pages()
        except pkv.PkvError:
            pass
    if w.shared_prefix:
        # every request forks from request 0's prompt pages, then leases its own suffix
        sp = w.shared_prefix // w.P
        reqs[0].lease_pages(sp)
        for b in range(1, w.B):
            reqs[b].close()
            reqs[b] = reqs[0].fork()
        for b, r in enumerate(reqs):
            r.lease_pages(int(w.n_pages[b]) - sp)
    else:
        for b, r in enumerate(reqs):
            r.release_pages()
            r.lease_pages(int(w.n_pages[b]))
    max_pages = int(w.n_pages.max())
    tables = np.full((w.B, max_pages), -1, dtype=np.int32)
    for b, r in enumerate(reqs):
        t = r.page_table()
        tables[b, :len(t)] = t
    k_pages, v_pages = pool.kv_pages(0)
    fill_history(k_pages, v_pages, w, tables, 0)
    q, k_new, v_new = step_inputs(w, 0)
    host = dict(q=q, k=k_new, v=v_new, tables=tables, lens=w.seq_lens.astype(np.int32))
    dev = dict(q=to_device(q), k=to_device(k_new), v=to_device(v_new),
               tables=torch.from_numpy(tables).cuda(), lens=torch.from_numpy(host["lens"]).cuda())
    max_seq_len = int(w.seq_lens.max())
    ws = pool.workspace(w.B, max_seq_len)
    out = torch.empty((w.B, w.HQ, w.D), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    return pool, reqs, host, dev, ws, out, max_seq_len


def run_gpu(args, compact=False):
    """The decode step of args.workload; with compact=True (a further workload measured
    in the same run) a short record without the end-to-end leg."""
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    rank, world = dist_init("nccl")
    w = make_workload(args.workload, rank, args.requests)
    pool, reqs, host, dev, ws, out, max_seq_len = setup_device(w, torch, args.cuda_cores)
    stream = torch.cuda.current_stream()
    shared = 0 if args.plain else int(w.shared_prefix)
    if shared:
        import ctypes
        import paged_kv_cache_decode_gb300 as pkv
        n = ctypes.c_size_t()
        pkv.check(pkv.lib.pkv_workspace_size_shared(pool.handle, w.B, max_seq_len, shared,
                                                    ctypes.byref(n)), "pkv_workspace_size_shared")
        ws = torch.empty(max(n.value, 16), dtype=torch.uint8, device="cuda")

    def step():
        if shared:
            pool.paged_decode_attention_shared(0, dev["q"], dev["k"], dev["v"], dev["tables"],
                                               dev["lens"], max_seq_len, shared, out=out,
                                               workspace=ws)
        else:
            pool.paged_decode_attention(0, dev["q"], dev["k"], dev["v"], dev["tables"], dev["lens"],
                                        max_seq_len, out=out, workspace=ws)

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert pool.check_device_status() == 0

    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for i in range(K):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    step_ms = start.elapsed_time(end) / K
    step_ms_max = max_over_ranks(step_ms, "cuda")

    # the split kernel alone: events recorded right before and after its launch
    # (a separate loop: the events sit between the plan and split kernels and
    # would hold back the split kernel's early launch in the timed step)
    evb = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    eva = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        pool.set_timing_events(evb[i], eva[i])
        step()
    torch.cuda.synchronize()
    pool.set_timing_events(None, None)
    kernel_ms = float(np.mean([b.elapsed_time(a) for b, a in zip(evb, eva)]))
    assert pool.check_device_status() == 0
    if compact:
        if sampler:
            sampler.stop()
        alg = algorithmic_bytes(w)
        peak, peak_kind = measured_peak_hbm()
        achieved = alg / (kernel_ms * 1e-3) / 1e9
        rec = {"workload": describe(w), "value": round(alg / (step_ms_max * 1e-3) / 1e9, 2),
               "unit": "GB/s", "steps": K, "warmup": args.warmup,
               "ms_per_step": round(step_ms_max, 5), "alg_bytes_per_step": alg,
               "tokens_per_s": round(w.B / (step_ms_max * 1e-3), 1),
               "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                            "unit": "GB/s", "frac": round(achieved / peak, 4),
                            "traffic": measured_traffic(w.name), "kernel": pool.kernel_name(),
                            "kernel_ms": round(kernel_ms, 5),
                            "peak_kind": peak_kind + " (hbm_gbs copy)"},
               "gpu_launches": 2 * K,
               "clocks": sampler.summary(t0, t1) if sampler else None}
        pool.close()
        return rec, w

    # end to end: host buffers in pinned memory, copies inside the timed region
    hp = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in host.items()
          if k in ("q", "tables", "lens")}
    for k in ("k", "v"):
        t = torch.from_numpy(host[k])
        hp[k] = (t.view(torch.int16) if host[k].dtype == np.uint16 else t).pin_memory()
    hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    dk = dev["k"].view(torch.int16) if dev["k"].dtype == torch.bfloat16 else dev["k"]
    dv = dev["v"].view(torch.int16) if dev["v"].dtype == torch.bfloat16 else dev["v"]
    h2d = sum(x.numel() * x.element_size() for x in hp.values())
    d2h = hout.numel() * hout.element_size()

    def e2e_step():
        dev["q"].copy_(hp["q"], non_blocking=True)
        dk.copy_(hp["k"], non_blocking=True)
        dv.copy_(hp["v"], non_blocking=True)
        dev["tables"].copy_(hp["tables"], non_blocking=True)
        dev["lens"].copy_(hp["lens"], non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)

    for _ in range(max(args.warmup, 3)):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(K):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K, "cuda")
    assert pool.check_device_status() == 0
    if sampler:
        sampler.stop()

    alg = algorithmic_bytes(w)
    kernel_name = pool.kernel_name()
    if shared:
        kernel_name = f"shared_prefix_kernel<{w.D}> + {kernel_name} + combine_kernel"
    line = None
    if rank == 0:
        peak, peak_kind = measured_peak_hbm()
        achieved = alg / (kernel_ms * 1e-3) / 1e9
        value = world * alg / (step_ms_max * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(step_ms_max, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.elem_bytes == 2 else "f32", "data": "synthetic",
            "config": decode_config(w, world, shared),
            "pct_of_8TBps": round(100 * value / world / NOMINAL_HBM_GBS, 2),
            "logical_GBps": round(world * logical_bytes(w) / (step_ms_max * 1e-3) / 1e9, 2),
            "tokens_per_s": round(world * w.B / (step_ms_max * 1e-3), 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": (measured_traffic(w.name, "shared_prefix",
                                                      [DECODE_SRC, SHARED_SRC]) if shared
                                     else measured_traffic(w.name)),
                         "kernel": kernel_name,
                         "kernel_ms": round(kernel_ms, 5), "peak_kind": peak_kind + " (hbm_gbs copy)"},
            "e2e": {"value": round(world * alg / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": K * (4 if shared else 2),
            "clocks": sampler.summary(t0, t1) if sampler else None,
        }
    pool.close()
    return line, w


# ------------------------------------------- the GPU arm, one request --

def token_bytes(w, t: int) -> int:
    """Algorithmic bytes of one token at retained length t through every layer."""
    es = w.elem_bytes
    per_layer = ((t - 1) * w.H * w.D * 2 * es + w.H * w.D * es * 2 * 2 + w.HQ * w.D * 4 * 2
                 + ((t + w.P - 1) // w.P) * 4)
    return w.layers * per_layer


def run_gpu_serial(args):
    """Single request through the transactional API: history built by serial
    begin / append x layers / commit up to t - 1; each timed step is one token at
    retained length t: begin_token, append_and_attend on every layer, abort_token
    (so every step sees the same t; commit is the same O(1) host update)."""
    import torch
    import paged_kv_cache_decode_gb300 as pkv
    import synth
    from synth import KHIST, VHIST, Q, F32
    from synth.device import to_device
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    rank, world = dist_init("nccl")
    w = make_workload(args.workload, rank)
    t = int(w.seq_lens[0])
    dt = "f32" if w.elem_bytes == 4 else "bf16"
    pool = pkv.Pool(w.layers, w.pool_pages, w.H, w.D, w.P, dt, w.max_context, w.seed,
                    query_heads=w.HQ)
    req = pool.request()
    out = torch.empty((w.HQ, w.D), dtype=torch.float32, device="cuda")

    def layer_inputs(pos):
        return [(to_device(synth.lane_rows(w.seed, Q, l, 0, w.HQ, pos, w.D, F32)),
                 to_device(synth.lane_rows(w.seed, KHIST, l, 0, w.H, pos, w.D, w.dtype)),
                 to_device(synth.lane_rows(w.seed, VHIST, l, 0, w.H, pos, w.D, w.dtype)))
                for l in range(w.layers)]

    for pos in range(t - 1):                      # history, untimed
        req.begin_token()
        for l, (q, k, v) in enumerate(layer_inputs(pos)):
            req.append_and_attend(l, q, k, v, out)
        req.commit_token()
    torch.cuda.synchronize()
    assert req.length == t - 1 and pool.check_device_status() == 0
    inputs = layer_inputs(t - 1)
    stream = torch.cuda.current_stream()

    # the timed token runs through the C ABI with the tensors' pointers taken once,
    # so it times the library's calls rather than the Python binding's argument
    # checks (the end-to-end leg below goes through the binding)
    import ctypes
    lib, h = pkv.lib, req.handle
    ptrs = [tuple(ctypes.c_void_p(x.data_ptr()) for x in layer) for layer in inputs]
    optr = ctypes.c_void_p(out.data_ptr())
    sptr = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    pos = ctypes.c_int64()

    def step():
        pkv.check(lib.pkv_begin_token(h, ctypes.byref(pos)), "pkv_begin_token")
        for l, (qp, kp, vp) in enumerate(ptrs):
            pkv.check(lib.pkv_append_and_attend(h, l, qp, kp, vp, optr, sptr),
                      "pkv_append_and_attend")
        pkv.check(lib.pkv_abort_token(h), "pkv_abort_token")

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for _ in range(K):
        step()
    t_issued = time.time()            # the host has issued every call
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    tok_ms = max_over_ranks(start.elapsed_time(end) / K, "cuda")
    host_us = (t_issued - t0) / K * 1e6
    # split kernel of one layer, alone
    evb = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    eva = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        pool.set_timing_events(evb[i], eva[i])
        req.begin_token()
        req.append_and_attend(0, *inputs[0], out)
        req.abort_token()
    torch.cuda.synchronize()
    pool.set_timing_events(None, None)
    kernel_ms = float(np.mean([b.elapsed_time(a) for b, a in zip(evb, eva)]))
    # end to end: the token's q, k, v of every layer copied in from pinned host memory
    # (one copy of one buffer), the calls through the C ABI on device pointers into it,
    # and every layer's output copied back (one copy)
    offs, pos_b = [], 0
    for layer in inputs:
        row = []
        for x in layer:
            row.append(pos_b)
            pos_b += (x.numel() * x.element_size() + 255) // 256 * 256
        offs.append(row)
    hin = torch.zeros(pos_b, dtype=torch.uint8).pin_memory()
    for layer, row in zip(inputs, offs):
        for x, o in zip(layer, row):
            n = x.numel() * x.element_size()
            hin[o:o + n].copy_(x.reshape(-1).view(torch.uint8).cpu())
    din = torch.empty(pos_b, dtype=torch.uint8, device="cuda")
    hout = torch.empty((w.layers, w.HQ, w.D), dtype=torch.float32).pin_memory()
    outs = torch.empty((w.layers, w.HQ, w.D), dtype=torch.float32, device="cuda")
    eptrs = [tuple(ctypes.c_void_p(din.data_ptr() + o) for o in row) for row in offs]
    optrs = [ctypes.c_void_p(outs[l].data_ptr()) for l in range(w.layers)]

    def e2e_step():
        din.copy_(hin, non_blocking=True)
        pkv.check(lib.pkv_begin_token(h, ctypes.byref(pos)), "pkv_begin_token")
        for l, (qp, kp, vp) in enumerate(eptrs):
            pkv.check(lib.pkv_append_and_attend(h, l, qp, kp, vp, optrs[l], sptr),
                      "pkv_append_and_attend")
        pkv.check(lib.pkv_abort_token(h), "pkv_abort_token")
        hout.copy_(outs, non_blocking=True)

    for _ in range(max(args.warmup, 3)):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K, "cuda")
    assert pool.check_device_status() == 0
    if sampler:
        sampler.stop()
    alg = token_bytes(w, t)
    kernel_name = pool.kernel_name()
    layer_alg = alg // w.layers
    h2d = sum(x.numel() * x.element_size() for layer in inputs for x in layer)
    line = None
    if rank == 0:
        peak, peak_kind = measured_peak_hbm()
        achieved = layer_alg / (kernel_ms * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": round(world * alg / (tok_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(tok_ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.elem_bytes == 2 else "f32", "data": "synthetic",
            "config": serial_config(w, world),
            "us_per_token": round(tok_ms * 1e3, 2),
            "host_issue_us_per_token": round(host_us, 2),
            "tokens_per_s": round(world / (tok_ms * 1e-3), 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": None,
                         "kernel": kernel_name,
                         "kernel_ms": round(kernel_ms, 5), "peak_kind": peak_kind + " (hbm_gbs copy)",
                         "note": "one layer's split kernel; latency-bound at this size"},
            "e2e": {"value": round(world * alg / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
                    "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": hout.numel() * 4},
            "gpu_launches": K * w.layers,     # one split kernel per layer (no plan kernel)
            "clocks": sampler.summary(t0, t1) if sampler else None,
        }
    pool.close()
    return line, w


# ------------------------------------------------- the GPU arm, prefill --

def prefill_flops(w) -> int:
    """Algorithmic FLOPs of one batched prefill: S = Q K^T and O = P V over every
    (query row, attended key) pair, 2 x d_h each."""
    from synth.workloads import attended_pairs
    return attended_pairs(w) * 4 * w.D


def measured_peak_bf16():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def setup_prefill(w, torch):
    """Pool, tables from the library's allocator, cached tokens in HBM, chunk inputs on device."""
    import paged_kv_cache_decode_gb300 as pkv
    from synth.device import fill_history, prefill_inputs, to_device
    pool = pkv.Pool(w.layers, w.pool_pages, w.H, w.D, w.P, "bf16" if w.elem_bytes == 2 else "f32",
                    w.max_context, w.seed,
                    query_heads=w.HQ, window=w.window)
    reqs = [pool.request() for _ in range(w.B)]
    for b, r in enumerate(reqs):
        r.lease_pages(int(w.n_pages[b]))
    tables = np.full((w.B, int(w.n_pages.max())), -1, dtype=np.int32)
    for b, r in enumerate(reqs):
        t = r.page_table()
        tables[b, :len(t)] = t
    k_pages, v_pages = pool.kv_pages(0)
    fill_history(k_pages, v_pages, w, tables, 0)
    q, k_new, v_new, cu = prefill_inputs(w, 0)
    host = dict(q=q, k=k_new, v=v_new, cu=cu, tables=tables, lens=w.seq_lens.astype(np.int32))
    dev = {k: (to_device(v) if v.dtype == np.uint16 else torch.from_numpy(v).cuda())
           for k, v in host.items()}
    N = int(cu[-1])
    out = torch.empty((N, w.HQ, w.D), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(pool.prefill_workspace_size(w.B, N), 16), dtype=torch.uint8,
                     device="cuda")
    torch.cuda.synchronize()
    return pool, reqs, host, dev, ws, out


def run_gpu_prefill(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    rank, world = dist_init("nccl")
    w = make_workload(args.workload, rank, args.requests)
    pool, reqs, host, dev, ws, out = setup_prefill(w, torch)
    stream = torch.cuda.current_stream()

    def step():
        pool.paged_prefill(0, dev["q"], dev["k"], dev["v"], dev["cu"], dev["tables"], dev["lens"],
                           out=out, workspace=ws)

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert pool.check_device_status() == 0

    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for _ in range(K):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    step_ms_max = max_over_ranks(start.elapsed_time(end) / K, "cuda")

    # the attention kernel alone, events recorded around its launch
    evb = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    eva = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        pool.set_timing_events(evb[i], eva[i])
        step()
    torch.cuda.synchronize()
    pool.set_timing_events(None, None)
    kernel_ms = float(np.mean([b.elapsed_time(a) for b, a in zip(evb, eva)]))

    # end to end: pinned host inputs copied in, the output copied out, every step
    hp = {}
    for k, v in host.items():
        t = torch.from_numpy(np.ascontiguousarray(v))
        hp[k] = (t.view(torch.int16) if v.dtype == np.uint16 else t).pin_memory()
    dv = {k: (d.view(torch.int16) if d.dtype == torch.bfloat16 else d) for k, d in dev.items()}
    hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in hp.values())
    d2h = hout.numel() * hout.element_size()

    def e2e_step():
        for k in hp:
            dv[k].copy_(hp[k], non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)

    for _ in range(max(args.warmup, 3)):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(K):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K, "cuda")
    assert pool.check_device_status() == 0
    if sampler:
        sampler.stop()

    flops = prefill_flops(w)
    N = int(host["cu"][-1])
    f32 = w.elem_bytes == 4
    if f32:
        # decode lanes: lane rows, block plan, the decode plan and the split kernel
        kernel = "split_decode_mma_kernel<f32,%d,8> (block lanes, table rows)" % w.D
        launches = 4
    else:
        kernel = "prefill_attention_kernel<%d>" % w.D
        launches = 3
    line = None
    if rank == 0:
        peak, peak_kind = measured_peak_bf16()
        peak_note = " (bf16_tflops burst, cuBLAS)"
        if f32:
            # tf32 products: the measured bf16 peak times the nominal tf32 / bf16 ratio
            peak, peak_note = round(peak * 1.1 / 2.25, 1), " (bf16_tflops burst x 1.1/2.25, tf32)"
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        value = world * flops / (step_ms_max * 1e-3) / 1e12
        line = {
            "metric": PREFILL_METRIC,
            "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(step_ms_max, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if f32 else "bf16", "data": "synthetic",
            "config": prefill_config(w, world),
            "tokens_per_s": round(world * N / (step_ms_max * 1e-3), 1),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                         "traffic": (None if f32 else
                                     measured_traffic(w.name, "prefill_attention", PREFILL_SRC)),
                         "kernel": kernel,
                         "kernel_ms": round(kernel_ms, 5),
                         "peak_kind": peak_kind + peak_note},
            "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                    "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": K * launches,
            "clocks": sampler.summary(t0, t1) if sampler else None,
        }
    for r in reqs:
        r.close()
    pool.close()
    return line, w


def oracle_prefill_sample(w, target_flops: float = 5e10, threads=0):
    """The first chunk tokens of request 0, as many as make about target_flops of
    oracle work, with the request's cached pages; a callable runs the oracle once."""
    import oracle
    import synth
    from synth import KHIST, VHIST
    from synth.device import prefill_inputs
    q, k_new, v_new, cu = prefill_inputs(w, 0)
    t, nb = int(w.seq_lens[0]), int(w.new_tokens[0])
    L0 = t - nb
    m = 0
    work = 0.0
    while m < nb and work < target_flops:
        keys = L0 + m + 1
        work += (min(keys, w.window) if w.window else keys) * w.HQ * 4 * w.D
        m += 1
    n = (L0 + m + w.P - 1) // w.P
    kp = synth.history_pages(w.seed, KHIST, 0, 0, n, w.H, w.P, w.D, L0, w.dtype)
    vp = synth.history_pages(w.seed, VHIST, 0, 0, n, w.H, w.P, w.D, L0, w.dtype)
    table = np.arange(n, dtype=np.int32)[None, :]
    qf = synth.bf16_to_f32(q[:m]) if q.dtype == np.uint16 else q[:m]
    cu1 = np.array([0, m], dtype=np.int32)
    lens = np.array([L0 + m], dtype=np.int32)

    def run():
        return oracle.paged_prefill(kp.copy(), vp.copy(), qf, k_new[:m], v_new[:m], cu1, table, lens,
                                    w.dtype, group=w.group, window=w.window, threads=threads)
    return run, work, m, L0


def cpu_baseline_prefill(w):
    import oracle
    run, work, m, L0 = oracle_prefill_sample(w)
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    return {"value": round(work / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"request 0: the first {m} of its {int(w.new_tokens[0])} chunk tokens after "
                      f"{L0} cached ({work / 1e9:.1f} GFLOP), fp64 C oracle, one pass, {dt:.2f} s",
            "tokens_per_s": round(m / dt, 3)}


# ------------------------------------------------------------ CPU oracle --

def oracle_sample(w, requests, threads=0):
    """Host pool holding the given requests' pages (compact ids), the step's inputs
    for them, and a callable that runs the oracle once."""
    import oracle
    import synth
    from synth import KHIST, VHIST, F32
    from synth.device import step_inputs
    q, k_new, v_new = step_inputs(w, 0)
    npg = [int(w.n_pages[b]) for b in requests]
    total = sum(npg)
    sd = np.float32 if w.elem_bytes == 4 else np.uint16
    kp = np.empty((total, w.H, w.P, w.D), dtype=sd)
    vp = np.empty_like(kp)
    tab = np.full((len(requests), max(npg)), -1, dtype=np.int32)
    off = 0
    for i, (b, n) in enumerate(zip(requests, npg)):
        t = int(w.seq_lens[b])
        tab[i, :n] = np.arange(off, off + n, dtype=np.int32)
        synth.history_pages(w.seed, KHIST, 0, b, n, w.H, w.P, w.D, t - 1, w.dtype, kp[off:off + n])
        synth.history_pages(w.seed, VHIST, 0, b, n, w.H, w.P, w.D, t - 1, w.dtype, vp[off:off + n])
        off += n
    lens = w.seq_lens[requests].astype(np.int32)
    dt = F32 if w.elem_bytes == 4 else 1

    def run():
        return oracle.paged_decode_attention(kp, vp, q[requests], k_new[requests], v_new[requests],
                                             tab, lens, dt, threads=threads, group=w.group,
                                             window=w.window)
    attended = np.minimum(lens.astype(np.int64), w.window) if w.window else lens.astype(np.int64)
    sample_bytes = int((attended - 1).sum()) * w.H * w.D * 2 * w.elem_bytes
    return run, sample_bytes, lens


def sample_requests(w, target_tokens: int):
    """Requests 0, 1, ... until their retained tokens reach target_tokens."""
    out, tok = [], 0
    for b in range(w.B):
        out.append(b)
        tok += int(w.seq_lens[b])
        if tok >= target_tokens:
            break
    return out


def sample_lanes(w, lanes: int):
    """Requests 0, 1, ... until they hold at least `lanes` (request, KV head) lanes."""
    return list(range(min(w.B, max(1, -(-lanes // w.H)))))


def attended_tokens(w, requests=None) -> int:
    lens = w.seq_lens.astype(np.int64)
    if requests is not None:
        lens = lens[list(requests)]
    if w.window:
        lens = np.minimum(lens, w.window)
    return int(lens.sum())


def oracle_decode_rate(w, requests, threads=0, passes=1):
    """The oracle on the given requests' lanes: the metric's value for the whole step
    (the step's algorithmic bytes over the time the sample's share of its work takes),
    the seconds of one pass, and the fraction of the step the sample is."""
    run, _, lens = oracle_sample(w, requests, threads=threads)
    t0 = time.perf_counter()
    for _ in range(passes):
        run()
    dt = (time.perf_counter() - t0) / passes
    frac = attended_tokens(w, requests) / attended_tokens(w)
    return algorithmic_bytes(w) * frac / dt / 1e9, dt, frac, lens


def cpu_baseline(w, lane_tokens=1 << 24):
    """The oracle on the whole step, or on its first requests up to ``lane_tokens``
    retained (lane, token) pairs (~10-30 s of CPU work on 16 cores); also one
    request on a single thread."""
    import oracle
    reqs = sample_requests(w, max(1, lane_tokens // w.H))
    value, dt, frac, lens = oracle_decode_rate(w, reqs)
    one = sample_lanes(w, 1)
    v1, dt1, _, lens1 = oracle_decode_rate(w, one, threads=1)
    return {"value": round(value, 4), "unit": "GB/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{len(reqs)} of {w.B} requests ({len(reqs) * w.H} lanes, "
                      f"{int(lens.sum())} tokens, {100 * frac:.1f} % of the step's work), fp64 C "
                      f"oracle, one pass, {dt:.2f} s; value = the step's algorithmic bytes over "
                      "the time of the whole step at that rate",
            "tokens_per_s": round(len(reqs) / dt, 3),
            "single_thread": {"value": round(v1, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"request 0 ({w.H} lanes, {int(lens1.sum())} tokens), "
                                        f"one thread, one pass, {dt1:.2f} s"}}


def run_reference_prefill(args, w, world):
    import oracle
    run, work, m, L0 = oracle_prefill_sample(w, target_flops=1e9)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = round(work / dt / 1e12, 6)
    sample = (f"each step: request 0's first {m} chunk tokens after {L0} cached "
              f"({work / 1e9:.1f} GFLOP), fp64 C oracle on the host cores; value = FLOPs of "
              "the sample over its time")
    return {
        "impl": "reference",
        "metric": PREFILL_METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": prefill_config(w, world),
        "tokens_per_s": round(m / dt, 3),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }, w


REFERENCE_BUDGET_S = 120.0      # host time the reference arm's timed and warm-up steps may take


def run_reference(args):
    """The oracle as it stands, on the host cores, on this arm's workload, metric and
    config.  Each step runs it over the step's first requests: at least as many lanes
    as the oracle has threads, more while the --steps + --warmup passes stay within
    REFERENCE_BUDGET_S (by a timed pass of the smallest sample), the whole step when
    that fits."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None, None
    import oracle
    w = make_workload(args.workload, 0, args.requests)
    if w.new_tokens is not None:
        return run_reference_prefill(args, w, world)
    cores = oracle.max_threads()
    reqs = sample_lanes(w, cores)
    run, _, _ = oracle_sample(w, reqs)
    t0 = time.perf_counter()
    run()
    per_token = (time.perf_counter() - t0) / attended_tokens(w, reqs)
    budget = REFERENCE_BUDGET_S / (args.steps + args.warmup)
    while len(reqs) < w.B and per_token * attended_tokens(w, reqs + [len(reqs)]) <= budget:
        reqs.append(len(reqs))
    if args.workload.startswith("single"):
        cfg = serial_config(w, world)
        alg = token_bytes(w, int(w.seq_lens[0]))
    else:
        cfg = decode_config(w, world, 0 if args.plain else int(w.shared_prefix))
        alg = algorithmic_bytes(w)
    run, _, lens = oracle_sample(w, reqs)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    frac = attended_tokens(w, reqs) / attended_tokens(w) / w.layers
    value = round(alg * frac / dt / 1e9, 4)
    sample = (f"each step: requests 0..{len(reqs) - 1} of {w.B} ({len(reqs) * w.H} lanes, "
              f"{int(lens.sum())} tokens, one layer: {100 * frac:.1f} % of the step's work), "
              f"fp64 C oracle on {cores} host threads; value = the step's algorithmic bytes over "
              "the time of the whole step at that rate")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / frac * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
        "tokens_per_s": round(w.B * frac / dt, 3),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line, w


# ------------------------------------------------------------------ main --

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="long")
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cuda-cores", action="store_true",
                    help="CUDA-core kernel even where the tensor-core kernel applies")
    ap.add_argument("--plain", action="store_true",
                    help="shared-prompt workload through the plain batched call")
    ap.add_argument("--requests", type=int, default=0,
                    help="keep only the first N requests (small profiling captures)")
    ap.add_argument("--no-extras", action="store_true",
                    help="long-context run without the batched and ragged records")
    return ap.parse_args(argv)


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        # the oracle and the input generator only; the library is neither built nor loaded
        import oracle
        import synth
        synth.build()
        oracle.build()
        line, _ = run_reference(args)
    else:
        import __graft_entry__
        __graft_entry__.build()
        if args.workload.startswith("single"):
            runner = run_gpu_serial
        elif args.workload.startswith("prefill"):
            runner = run_gpu_prefill
        else:
            runner = run_gpu
        line, w = runner(args)
        rank, world, _ = dist_env()
        if line is not None and world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = (cpu_baseline_prefill(w) if w.new_tokens is not None
                                    else cpu_baseline(w))
        if (line is not None and world == 1 and args.workload == "long" and not args.requests
                and not args.no_extras):
            extra = {}
            for name in EXTRA_WORKLOADS:
                sub = argparse.Namespace(**vars(args))
                sub.workload, sub.steps = name, min(args.steps, 100)
                extra[name], _ = run_gpu(sub, compact=True)
            line["also_measured"] = extra
            line["gpu_launches"] += sum(r["gpu_launches"] for r in extra.values())
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
