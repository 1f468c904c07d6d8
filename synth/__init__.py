"""Seeded synthetic inputs shared by the fp64 oracle and the device harness.

This package is input plumbing only.  It holds no attention arithmetic: it
draws q / k / v / history values (counter-based SplitMix64, see ``synth.c``),
request lengths and allocator operation sequences, so that the oracle and the
CUDA path are fed identical bytes.  Values for logical token ``j`` of head
``h`` of request ``b`` in layer ``l`` are a pure function of
``(seed, kind, l, b, h, j, d)``; where that token lands in the paged pool is
decided by the page tables, not by the generator.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynth.so")
_lock = threading.Lock()
_lib = None

# kinds of value streams
KHIST = 0   # key rows; token j of a request's key sequence (history and new)
VHIST = 1   # value rows
Q = 2       # query rows

F32 = 0
BF16 = 1

MASK64 = (1 << 64) - 1


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_build/libsynth.so`` (gcc, OpenMP if present)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
            L.synth_splitmix64_at.restype = u64
            L.synth_splitmix64_at.argtypes = [u64, u64]
            L.synth_stream_seed.restype = u64
            L.synth_stream_seed.argtypes = [u64, u64]
            L.synth_rows.restype = None
            L.synth_rows.argtypes = [u64, u64, i64, i64, i64, i64, ctypes.c_int, vp]
            L.synth_history_pages.restype = None
            L.synth_history_pages.argtypes = [u64, u64, i64, i64, i64, i64, i64, ctypes.c_int, vp]
            L.synth_history_pages_from.restype = None
            L.synth_history_pages_from.argtypes = [u64, u64, i64, i64, i64, i64, i64, i64,
                                                   ctypes.c_int, vp]
            L.synth_f32_to_bf16_array.restype = None
            L.synth_f32_to_bf16_array.argtypes = [vp, i64, vp]
            L.synth_max_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def stream_id(kind: int, layer: int, request: int) -> int:
    """Stream of one (kind, layer, request)."""
    return ((request * 4096 + layer) * 8 + kind) & MASK64


def splitmix64_at(seed: int, i: int) -> int:
    return int(lib().synth_splitmix64_at(seed & MASK64, i & MASK64))


def _np_dtype(dtype: int):
    return np.float32 if dtype == F32 else np.uint16


def rows(seed: int, kind: int, layer: int, request: int, head: int, token0: int,
         nrows: int, D: int, dtype: int = F32) -> np.ndarray:
    """Rows ``token0 .. token0+nrows-1`` of one (kind, layer, request, head): [nrows, D]."""
    out = np.empty((nrows, D), dtype=_np_dtype(dtype))
    if nrows > 0:
        lib().synth_rows(seed & MASK64, stream_id(kind, layer, request), head, token0, nrows, D,
                         dtype, out.ctypes.data)
    return out


def lane_rows(seed: int, kind: int, layer: int, request: int, H: int, token: int, D: int,
              dtype: int = F32) -> np.ndarray:
    """Row ``token`` of every head of one request: [H, D]."""
    return np.stack([rows(seed, kind, layer, request, h, token, 1, D, dtype)[0] for h in range(H)])


def history_pages(seed: int, kind: int, layer: int, request: int, n_pages: int, H: int, P: int,
                  D: int, n_tokens: int, dtype: int, out: np.ndarray | None = None,
                  first_page: int = 0) -> np.ndarray:
    """Physical-layout pages [n_pages, H, P, D] holding logical pages first_page ..
    first_page + n_pages - 1 of tokens ``0 .. n_tokens-1`` (rest zero)."""
    if out is None:
        out = np.empty((n_pages, H, P, D), dtype=_np_dtype(dtype))
    assert out.shape == (n_pages, H, P, D) and out.dtype == _np_dtype(dtype)
    assert out.flags["C_CONTIGUOUS"]
    if n_pages > 0:
        lib().synth_history_pages_from(seed & MASK64, stream_id(kind, layer, request), first_page,
                                       n_pages, H, P, D, n_tokens, dtype, out.ctypes.data)
    return out


def request_history_pages(w, kind: int, layer: int, request: int, n_pages: int, n_tokens: int,
                          out: np.ndarray | None = None) -> np.ndarray:
    """History pages of one request of workload w.  With a shared prefix of S tokens
    (w.shared_prefix, a multiple of the page size), tokens j < S are request 0's: every
    request decodes after the same prompt."""
    S = getattr(w, "shared_prefix", 0)
    if out is None:
        out = np.empty((n_pages, w.H, w.P, w.D), dtype=_np_dtype(w.dtype))
    sp = min(S // w.P, n_pages) if request != 0 else 0
    if sp:
        history_pages(w.seed, kind, layer, 0, sp, w.H, w.P, w.D, n_tokens, w.dtype, out[:sp])
    if n_pages > sp:
        history_pages(w.seed, kind, layer, request, n_pages - sp, w.H, w.P, w.D, n_tokens, w.dtype,
                      out[sp:], first_page=sp)
    return out


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().synth_f32_to_bf16_array(x.ctypes.data, x.size, out.ctypes.data)
    return out


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 (exact)."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def host_threads() -> int:
    return int(lib().synth_max_threads())


class SplitMix64:
    """Sequential SplitMix64 stream (pure Python), for small host-side draws."""

    def __init__(self, seed: int):
        self.state = seed & MASK64

    def next(self) -> int:
        self.state = (self.state + 0x9E3779B97F4A7C15) & MASK64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        return z ^ (z >> 31)
