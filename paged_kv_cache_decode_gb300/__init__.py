"""Paged KV-cache decode attention for NVIDIA GB300 (sm_103a).

Thin Python layer over libpkv.so (C ABI in include/pkv.h).  PyTorch supplies
device memory and streams; the kernels do all the work.  Names follow the C
ABI without its ``pkv_`` prefix:

    pool = pool_create(layers, pages, heads, head_dim, page_size=16, dtype="bf16",
                       max_context=4096, seed=0)
    req = request_create(pool)
    pos = begin_token(req)                       # reserve the next position
    out = append_and_attend(req, layer, q, k, v) # once per layer, [H, d_h] each
    commit_token(req)                            # or abort_token(req)

    paged_decode_attention(pool, layer, q, k_new, v_new, page_tables, seq_lens,
                           max_seq_len, out=out, workspace=ws)   # batched

The operations follow "Incremental Serving" (sections "Request flow" and
"Paged KV-cache layout") and the attention arithmetic of "38 · Cached
generation" (function incremental_mixture).
"""
from __future__ import annotations

import ctypes

import torch

from .binding import (  # noqa: F401
    lib, check, PkvError, pkv_counters, pkv_pool_options, LIB_PATH,
    PKV_OK, PKV_ERR_INVALID_ARGUMENT, PKV_ERR_OUT_OF_PAGES, PKV_ERR_CAPACITY_EXCEEDED,
    PKV_ERR_BAD_STATE, PKV_ERR_OUT_OF_MEMORY, PKV_ERR_CUDA, PKV_ERR_DEVICE_CHECK,
    PKV_ERR_NO_STORAGE, PKV_ERR_UNSUPPORTED, PKV_F32, PKV_BF16, PKV_POOL_HOST_ONLY,
    PKV_POOL_CUDA_CORES,
    PKV_DEVERR_SEQ_LEN, PKV_DEVERR_PAGE_ID, PKV_DEVERR_TIMEOUT, PKV_DEVERR_SHARED,
    PKV_INJECT_NONE, PKV_INJECT_LEASE, PKV_INJECT_LAYER, PKV_INJECT_DEVICE_WAIT,
)

__all__ = [
    "Pool", "Request", "PkvError", "pool_create", "pool_destroy", "request_create",
    "request_destroy", "request_fork", "lease_pages", "release_pages", "begin_token", "append_and_attend",
    "commit_token", "abort_token", "begin_chunk", "prefill_chunk", "paged_decode_attention",
    "paged_decode_attention_shared",
    "paged_prefill", "workspace_size",
    "check_device_status", "PKV_F32", "PKV_BF16",
]

_TORCH_DTYPE = {PKV_F32: torch.float32, PKV_BF16: torch.bfloat16}


def _dtype_code(dtype) -> int:
    if dtype in (PKV_F32, "f32", "fp32", "float32", torch.float32):
        return PKV_F32
    if dtype in (PKV_BF16, "bf16", "bfloat16", torch.bfloat16):
        return PKV_BF16
    raise ValueError(f"unsupported storage dtype {dtype!r}")


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor, name: str, dtype, shape) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


class _DeviceArray:
    """__cuda_array_interface__ view of library-owned device memory."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


class Pool:
    """A paged K/V pool: per layer, key and value pages [pages, heads, page_size, head_dim].

    ``heads`` is the number of KV heads stored per page; ``query_heads`` (default:
    ``heads``) the heads of the query and output, a multiple of ``heads``
    (grouped-query attention); ``window`` > 0 limits every query to the last
    ``window`` positions (sliding window)."""

    def __init__(self, layers: int, pages: int, heads: int, head_dim: int, page_size: int = 16,
                 dtype="f32", max_context: int = 4096, seed: int = 0, host_only: bool = False,
                 query_heads: int = 0, cuda_cores: bool = False, window: int = 0):
        self.layers, self.heads, self.head_dim, self.page_size = layers, heads, head_dim, page_size
        self.query_heads = query_heads or heads
        self.window = window
        self.dtype = _dtype_code(dtype)
        self.torch_dtype = _TORCH_DTYPE[self.dtype]
        self.max_context = max_context
        self.host_only = host_only
        o = pkv_pool_options()
        check(lib.pkv_pool_options_init(ctypes.byref(o)), "pkv_pool_options_init")
        o.layers, o.pages, o.kv_heads, o.query_heads = layers, pages, heads, self.query_heads
        o.head_dim, o.page_size, o.dtype, o.max_context = head_dim, page_size, self.dtype, max_context
        o.seed = seed & ((1 << 64) - 1)
        o.window = window
        o.flags = (PKV_POOL_HOST_ONLY if host_only else 0) | (PKV_POOL_CUDA_CORES if cuda_cores else 0)
        h = ctypes.c_void_p()
        check(lib.pkv_pool_create_ex(ctypes.byref(o), ctypes.byref(h)), "pkv_pool_create_ex")
        self._h = h
        self.pages = self.page_info()[0]
        self.max_pages_per_request = -(-max_context // page_size)
        self._requests = []
        self._ws = {}

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None:
            raise ValueError("pool is closed")
        return self._h

    # -- storage ----------------------------------------------------------
    def kv_pages(self, layer: int):
        """(K, V) tensors viewing layer ``layer``'s device pages, [pages, H, P, D]."""
        k, v = ctypes.c_void_p(), ctypes.c_void_p()
        check(lib.pkv_pool_kv_ptr(self.handle, layer, ctypes.byref(k), ctypes.byref(v)),
              "pkv_pool_kv_ptr")
        shape = (self.pages, self.heads, self.page_size, self.head_dim)
        typestr = "<f4" if self.dtype == PKV_F32 else "<i2"
        out = []
        for ptr in (k.value, v.value):
            t = torch.as_tensor(_DeviceArray(ptr, shape, typestr), device="cuda")
            out.append(t if self.dtype == PKV_F32 else t.view(torch.bfloat16))
        return tuple(out)

    @property
    def tensor_cores(self) -> bool:
        """True if this pool's attention runs the tensor-core kernel."""
        v = ctypes.c_int()
        check(lib.pkv_pool_kernel(self.handle, ctypes.byref(v)), "pkv_pool_kernel")
        return bool(v.value)

    def kernel_name(self) -> str:
        """The decode split kernel this pool launches (larger groups of query heads per
        KV head run as lanes of 16 on the bf16 tensor-core kernel, of 8 otherwise)."""
        g = self.query_heads // self.heads
        st = "f32" if self.dtype == PKV_F32 else "bf16"
        if self.tensor_cores:
            return f"split_decode_mma_kernel<{st},{self.head_dim},{min(g, 16 if st == 'bf16' else 8)}>"
        return f"split_decode_kernel<{st},{self.head_dim},{min(g, 8)}>"

    def bytes(self) -> int:
        b = ctypes.c_uint64()
        check(lib.pkv_pool_bytes(self.handle, ctypes.byref(b)), "pkv_pool_bytes")
        return b.value

    def page_info(self):
        n, f = ctypes.c_int64(), ctypes.c_int64()
        check(lib.pkv_pool_pages(self.handle, ctypes.byref(n), ctypes.byref(f)), "pkv_pool_pages")
        return n.value, f.value

    @property
    def free_pages(self) -> int:
        return self.page_info()[1]

    def free_list(self) -> list:
        n = ctypes.c_int64()
        check(lib.pkv_pool_free_list(self.handle, None, 0, ctypes.byref(n)), "pkv_pool_free_list")
        buf = (ctypes.c_int32 * max(n.value, 1))()
        check(lib.pkv_pool_free_list(self.handle, buf, n.value, ctypes.byref(n)),
              "pkv_pool_free_list")
        return list(buf[:n.value])

    # -- requests ---------------------------------------------------------
    def request(self) -> "Request":
        r = Request(self)
        self._requests.append(r)
        return r

    def page_refs(self, page: int) -> int:
        """Requests referencing physical page `page` (0: free)."""
        n = ctypes.c_int()
        check(lib.pkv_pool_page_refs(self.handle, page, ctypes.byref(n)), "pkv_pool_page_refs")
        return n.value

    # -- batched ----------------------------------------------------------
    def workspace_size(self, batch: int, max_seq_len: int) -> int:
        b = ctypes.c_size_t()
        check(lib.pkv_workspace_size(self.handle, batch, max_seq_len, ctypes.byref(b)),
              "pkv_workspace_size")
        return b.value

    def workspace(self, batch: int, max_seq_len: int, device=None) -> torch.Tensor:
        """A device scratch buffer of workspace_size bytes (uint8)."""
        n = self.workspace_size(batch, max_seq_len)
        return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")

    def paged_decode_attention(self, layer: int, q, k_new, v_new, page_tables, seq_lens,
                               max_seq_len: int, out=None, workspace=None, stream=None):
        B = q.shape[0]
        H, HQ, D = self.heads, self.query_heads, self.head_dim
        if out is None:
            out = torch.empty((B, HQ, D), dtype=torch.float32, device=q.device)
        if workspace is None:
            key = (B, max_seq_len)
            if key not in self._ws:
                self._ws[key] = self.workspace(B, max_seq_len, q.device)
            workspace = self._ws[key]
        if page_tables.dim() != 2 or page_tables.shape[0] != B:
            raise ValueError("page_tables must be [batch, max_pages]")
        check(lib.pkv_paged_decode_attention(
            self.handle, layer, B,
            _dev(q, "q", torch.float32, (B, HQ, D)),
            _dev(k_new, "k_new", self.torch_dtype, (B, H, D)),
            _dev(v_new, "v_new", self.torch_dtype, (B, H, D)),
            _dev(page_tables, "page_tables", torch.int32, None), page_tables.shape[1],
            _dev(seq_lens, "seq_lens", torch.int32, (B,)), int(max_seq_len),
            _dev(out, "out", torch.float32, (B, HQ, D)),
            _dev(workspace, "workspace", torch.uint8, None), workspace.numel(),
            _stream_ptr(stream)), "pkv_paged_decode_attention")
        return out

    def paged_decode_attention_shared(self, layer: int, q, k_new, v_new, page_tables, seq_lens,
                                      max_seq_len: int, shared_len: int, out=None, workspace=None,
                                      stream=None):
        """paged_decode_attention for a batch whose first shared_len positions share
        request 0's pages (read once per KV head)."""
        B = q.shape[0]
        H, HQ, D = self.heads, self.query_heads, self.head_dim
        if out is None:
            out = torch.empty((B, HQ, D), dtype=torch.float32, device=q.device)
        if workspace is None:
            key = ("shared", B, max_seq_len, shared_len)
            if key not in self._ws:
                n = ctypes.c_size_t()
                check(lib.pkv_workspace_size_shared(self.handle, B, int(max_seq_len), int(shared_len),
                                                    ctypes.byref(n)), "pkv_workspace_size_shared")
                self._ws[key] = torch.empty(max(n.value, 16), dtype=torch.uint8, device=q.device)
            workspace = self._ws[key]
        if page_tables.dim() != 2 or page_tables.shape[0] != B:
            raise ValueError("page_tables must be [batch, max_pages]")
        check(lib.pkv_paged_decode_attention_shared(
            self.handle, layer, B,
            _dev(q, "q", torch.float32, (B, HQ, D)),
            _dev(k_new, "k_new", self.torch_dtype, (B, H, D)),
            _dev(v_new, "v_new", self.torch_dtype, (B, H, D)),
            _dev(page_tables, "page_tables", torch.int32, None), page_tables.shape[1],
            _dev(seq_lens, "seq_lens", torch.int32, (B,)), int(max_seq_len), int(shared_len),
            _dev(out, "out", torch.float32, (B, HQ, D)),
            _dev(workspace, "workspace", torch.uint8, None), workspace.numel(),
            _stream_ptr(stream)), "pkv_paged_decode_attention_shared")
        return out

    def prefill_workspace_size(self, batch: int, total_new: int) -> int:
        n = ctypes.c_size_t()
        check(lib.pkv_prefill_workspace_size(self.handle, batch, total_new, ctypes.byref(n)),
              "pkv_prefill_workspace_size")
        return n.value

    def paged_prefill(self, layer: int, q, k_new, v_new, cu_new, page_tables, seq_lens, out=None,
                      workspace=None, stream=None):
        """Batched prefill of one layer: request b appends rows cu_new[b] .. cu_new[b+1]-1
        of q / k_new / v_new (the pool's storage dtype) after its seq_lens[b] - n_b cached
        tokens; returns out [N, query_heads, head_dim] fp32."""
        N = q.shape[0]
        B = cu_new.shape[0] - 1
        H, HQ, D = self.heads, self.query_heads, self.head_dim
        if out is None:
            out = torch.empty((N, HQ, D), dtype=torch.float32, device=q.device)
        if workspace is None:
            key = ("prefill", B, N)
            if key not in self._ws:
                n = self.prefill_workspace_size(B, N)
                self._ws[key] = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
            workspace = self._ws[key]
        if page_tables.dim() != 2 or page_tables.shape[0] != B:
            raise ValueError("page_tables must be [batch, max_pages]")
        check(lib.pkv_paged_prefill(
            self.handle, layer, B, N,
            _dev(q, "q", self.torch_dtype, (N, HQ, D)),
            _dev(k_new, "k_new", self.torch_dtype, (N, H, D)),
            _dev(v_new, "v_new", self.torch_dtype, (N, H, D)),
            _dev(cu_new, "cu_new", torch.int32, (B + 1,)),
            _dev(page_tables, "page_tables", torch.int32, None), page_tables.shape[1],
            _dev(seq_lens, "seq_lens", torch.int32, (B,)),
            _dev(out, "out", torch.float32, (N, HQ, D)),
            _dev(workspace, "workspace", torch.uint8, None), workspace.numel(),
            _stream_ptr(stream)), "pkv_paged_prefill")
        return out

    def set_timing_events(self, before, after) -> None:
        """Record two torch.cuda.Event around every later split (attention) kernel
        launch of this pool; (None, None) turns it off."""
        def handle(ev):
            if ev is None:
                return None
            if not ev.cuda_event:          # torch creates the event lazily
                ev.record()
            return ctypes.c_void_p(ev.cuda_event)
        check(lib.pkv_pool_set_timing_events(self.handle, handle(before), handle(after)),
              "pkv_pool_set_timing_events")

    def inject_fault(self, kind: int, arg: int = 0, wait_limit_ns: int = 0) -> None:
        """Arm a one-shot failure hook (PKV_INJECT_*; tests of the recovery paths)."""
        check(lib.pkv_pool_inject_fault(self.handle, kind, arg, wait_limit_ns),
              "pkv_pool_inject_fault")

    def check_device_status(self) -> int:
        """Synchronise; return the device error bits (raises PkvError if any were set)."""
        bits = ctypes.c_uint32()
        st = lib.pkv_check_device_status(self.handle, ctypes.byref(bits))
        if st not in (PKV_OK, PKV_ERR_DEVICE_CHECK):
            check(st, "pkv_check_device_status")
        if st == PKV_ERR_DEVICE_CHECK:
            raise PkvError(st, f"pkv_check_device_status (bits 0x{bits.value:x})")
        return bits.value

    def device_status_bits(self) -> int:
        """Synchronise; return and clear the device error bits without raising on them."""
        bits = ctypes.c_uint32()
        st = lib.pkv_check_device_status(self.handle, ctypes.byref(bits))
        if st not in (PKV_OK, PKV_ERR_DEVICE_CHECK):
            check(st, "pkv_check_device_status")
        return bits.value

    def close(self) -> None:
        if self._h is not None:
            for r in list(self._requests):
                r.close()
            check(lib.pkv_pool_destroy(self._h), "pkv_pool_destroy")
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


class Request:
    """One request's logical page table, visible length and pending token."""

    def __init__(self, pool: Pool, handle=None):
        self.pool = pool
        if handle is None:
            handle = ctypes.c_void_p()
            check(lib.pkv_request_create(pool.handle, ctypes.byref(handle)), "pkv_request_create")
        self._h = handle

    def fork(self) -> "Request":
        """A request sharing every page of this one (copy-on-write on later writes)."""
        h = ctypes.c_void_p()
        check(lib.pkv_request_fork(self.handle, ctypes.byref(h)), "pkv_request_fork")
        child = Request(self.pool, h)
        self.pool._requests.append(child)
        return child

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None:
            raise ValueError("request is closed")
        return self._h

    def lease_pages(self, n: int) -> None:
        check(lib.pkv_lease_pages(self.handle, n), "pkv_lease_pages")

    def release_pages(self) -> None:
        check(lib.pkv_release_pages(self.handle), "pkv_release_pages")

    @property
    def length(self) -> int:
        n = ctypes.c_int64()
        check(lib.pkv_request_length(self.handle, ctypes.byref(n)), "pkv_request_length")
        return n.value

    def page_table(self) -> list:
        n = ctypes.c_int64()
        check(lib.pkv_request_page_table(self.handle, None, 0, ctypes.byref(n)),
              "pkv_request_page_table")
        buf = (ctypes.c_int32 * max(n.value, 1))()
        check(lib.pkv_request_page_table(self.handle, buf, n.value, ctypes.byref(n)),
              "pkv_request_page_table")
        return list(buf[:n.value])

    def counters(self) -> dict:
        c = pkv_counters()
        check(lib.pkv_request_counters(self.handle, ctypes.byref(c)), "pkv_request_counters")
        return {"committed_tokens": c.committed_tokens, "cache_appends": c.cache_appends,
                "score_cells": c.score_cells}

    def begin_token(self) -> int:
        pos = ctypes.c_int64()
        check(lib.pkv_begin_token(self.handle, ctypes.byref(pos)), "pkv_begin_token")
        return pos.value

    def append_and_attend(self, layer: int, q, k, v, out=None, stream=None):
        """q [query_heads, d_h] fp32; k, v [heads, d_h] storage dtype; returns out
        [query_heads, d_h] fp32."""
        p = self.pool
        qshape = (p.query_heads, p.head_dim)
        kshape = (p.heads, p.head_dim)
        if out is None:
            out = torch.empty(qshape, dtype=torch.float32, device=q.device)
        check(lib.pkv_append_and_attend(
            self.handle, layer, _dev(q, "q", torch.float32, qshape),
            _dev(k, "k", p.torch_dtype, kshape), _dev(v, "v", p.torch_dtype, kshape),
            _dev(out, "out", torch.float32, qshape), _stream_ptr(stream)), "pkv_append_and_attend")
        return out

    def begin_chunk(self, n: int) -> int:
        """Open a chunk of n positions at the visible length; returns the first."""
        pos = ctypes.c_int64()
        check(lib.pkv_begin_chunk(self.handle, n, ctypes.byref(pos)), "pkv_begin_chunk")
        return pos.value

    def prefill_chunk(self, layer: int, q, k, v, out=None, stream=None):
        """One layer of the pending chunk: q [n, query_heads, d_h], k, v [n, heads, d_h]
        in the pool's storage dtype; returns out [n, query_heads, d_h] fp32."""
        p = self.pool
        n = q.shape[0]
        qshape = (n, p.query_heads, p.head_dim)
        kshape = (n, p.heads, p.head_dim)
        if out is None:
            out = torch.empty(qshape, dtype=torch.float32, device=q.device)
        check(lib.pkv_prefill_chunk(
            self.handle, layer, _dev(q, "q", p.torch_dtype, qshape),
            _dev(k, "k", p.torch_dtype, kshape), _dev(v, "v", p.torch_dtype, kshape),
            _dev(out, "out", torch.float32, qshape), _stream_ptr(stream)), "pkv_prefill_chunk")
        return out

    def commit_token(self) -> None:
        check(lib.pkv_commit_token(self.handle), "pkv_commit_token")

    def abort_token(self) -> None:
        check(lib.pkv_abort_token(self.handle), "pkv_abort_token")

    def close(self) -> None:
        if self._h is not None:
            check(lib.pkv_request_destroy(self._h), "pkv_request_destroy")
            self._h = None
            if self in self.pool._requests:
                self.pool._requests.remove(self)


# --------------------------------------------------------- C-ABI names --

def pool_create(layers, pages, heads, head_dim, page_size=16, dtype="f32", max_context=4096,
                seed=0, host_only=False, query_heads=0, cuda_cores=False, window=0) -> Pool:
    return Pool(layers, pages, heads, head_dim, page_size, dtype, max_context, seed, host_only,
                query_heads, cuda_cores, window)


def pool_destroy(pool: Pool) -> None:
    pool.close()


def request_create(pool: Pool) -> Request:
    return pool.request()


def request_destroy(req: Request) -> None:
    req.close()


def request_fork(parent: Request) -> Request:
    return parent.fork()


def lease_pages(req: Request, n: int) -> None:
    req.lease_pages(n)


def release_pages(req: Request) -> None:
    req.release_pages()


def begin_token(req: Request) -> int:
    return req.begin_token()


def append_and_attend(req: Request, layer, q, k, v, out=None, stream=None):
    return req.append_and_attend(layer, q, k, v, out, stream)


def begin_chunk(req: Request, n: int) -> int:
    return req.begin_chunk(n)


def prefill_chunk(req: Request, layer, q, k, v, out=None, stream=None):
    return req.prefill_chunk(layer, q, k, v, out, stream)


def commit_token(req: Request) -> None:
    req.commit_token()


def abort_token(req: Request) -> None:
    req.abort_token()


def workspace_size(pool: Pool, batch: int, max_seq_len: int) -> int:
    return pool.workspace_size(batch, max_seq_len)


def paged_decode_attention(pool: Pool, layer, q, k_new, v_new, page_tables, seq_lens, max_seq_len,
                           out=None, workspace=None, stream=None):
    return pool.paged_decode_attention(layer, q, k_new, v_new, page_tables, seq_lens, max_seq_len,
                                       out, workspace, stream)


def paged_decode_attention_shared(pool: Pool, layer, q, k_new, v_new, page_tables, seq_lens,
                                  max_seq_len, shared_len, out=None, workspace=None, stream=None):
    return pool.paged_decode_attention_shared(layer, q, k_new, v_new, page_tables, seq_lens,
                                              max_seq_len, shared_len, out, workspace, stream)


def paged_prefill(pool: Pool, layer, q, k_new, v_new, cu_new, page_tables, seq_lens, out=None,
                  workspace=None, stream=None):
    return pool.paged_prefill(layer, q, k_new, v_new, cu_new, page_tables, seq_lens, out,
                              workspace, stream)


def check_device_status(pool: Pool) -> int:
    return pool.check_device_status()
