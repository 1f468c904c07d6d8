"""ORACLE — test infrastructure only.

A plain, slow, obviously correct CPU restatement of paged decode attention
and of the page-pool / transaction bookkeeping around it, in fp64.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA path and imports
nothing from the product package; the only thing both sides share is the
seeded input generator package ``synth``.

* ``attention.c`` — the attention arithmetic (append, gather through the page
  table, fp64 scores, stable softmax, value mixture).
* ``model.py``    — the pool, free list, page tables and the transactional
  begin / append / commit / abort state machine, as a Python model.

Pins (tests under ``tests/`` marked ``not gpu``): brute-force causal
attention, contiguous single-page layout, physical-page permutation
invariance, closed forms (t = 1, q = 0, equal keys), transactional abort, the
score-cell counts printed by the sources, the KV-bytes worked example.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile ``attention.c`` into ``_build/liboracle.so`` (gcc; OpenMP if present)."""
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


def load(path: str):
    """Load an oracle library file and declare its entry points."""
    L = ctypes.CDLL(path)
    i32, i64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
    L.orc_append.restype = i32
    L.orc_append.argtypes = [i32, i32, i32, i32, i32, vp, vp, i64, vp, vp, vp, i32, vp]
    L.orc_paged_decode_attention.restype = i32
    L.orc_paged_decode_attention.argtypes = [i32, i32, i32, i32, i32, vp, vp, i64, vp, vp,
                                             vp, vp, i32, vp, vp, vp, i64, i32]
    L.orc_paged_decode_attention_ex.restype = i32
    L.orc_paged_decode_attention_ex.argtypes = [i32, i32, i32, i64, i32, i32, i32, vp, vp, i64, vp,
                                                vp, vp, vp, i32, vp, vp, vp, i64, i32]
    L.orc_paged_decode_attention_gqa.restype = i32
    L.orc_paged_decode_attention_gqa.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, i64, vp, vp,
                                                 vp, vp, i32, vp, vp, vp, i64, i32]
    L.orc_paged_prefill.restype = i32
    L.orc_paged_prefill.argtypes = [i32, i32, i32, i64, i32, i32, i32, vp, vp, i64, vp, vp, vp, vp,
                                    vp, i32, vp, vp, i32]
    L.orc_max_threads.restype = i32
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
    return _lib


def _storage_dtype(dtype: int):
    return np.float32 if dtype == F32 else np.uint16


def _check_pool(pool: np.ndarray, dtype: int):
    assert pool.dtype == _storage_dtype(dtype) and pool.ndim == 4 and pool.flags["C_CONTIGUOUS"]


def paged_decode_attention(k_pool: np.ndarray, v_pool: np.ndarray, q: np.ndarray,
                           k_new: np.ndarray, v_new: np.ndarray, tables: np.ndarray,
                           seq_lens: np.ndarray, dtype: int = F32, lanes=None,
                           threads: int = 0, library=None, group: int = 1,
                           window: int = 0) -> np.ndarray:
    """Append the new rows, then fp64 attention of each lane's newest query.

    k_pool, v_pool: one layer, [pages, H, P, D] storage dtype (fp32 or bf16 bits as
    uint16); modified in place by the append.  q [B, H*group, D] fp32; k_new, v_new
    [B, H, D] storage dtype; tables [B, max_pages] int32; seq_lens [B] int32 (t_b,
    new token included).  Query head qh reads KV head qh // group.  With window W > 0
    only the last W positions are attended.  Returns out
    [B, H*group, D] fp64 (query lanes b*H*group + qh not listed in ``lanes`` are
    left zero).  ``library``: an alternative loaded oracle library (tests only).
    """
    _check_pool(k_pool, dtype)
    _check_pool(v_pool, dtype)
    n_pages, H, P, D = k_pool.shape
    assert v_pool.shape == k_pool.shape
    q = np.ascontiguousarray(q, dtype=np.float32)
    B = q.shape[0]
    assert q.shape == (B, H * group, D)
    k_new = np.ascontiguousarray(k_new, dtype=_storage_dtype(dtype))
    v_new = np.ascontiguousarray(v_new, dtype=_storage_dtype(dtype))
    assert k_new.shape == (B, H, D) and v_new.shape == (B, H, D)
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    assert tables.ndim == 2 and tables.shape[0] == B
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    assert seq_lens.shape == (B,)
    out = np.zeros((B, H * group, D), dtype=np.float64)
    lane_arr = None
    n_lanes = 0
    if lanes is not None:
        lane_arr = np.ascontiguousarray(lanes, dtype=np.int64)
        n_lanes = lane_arr.size
    L = library or lib()
    if group == 1 and window == 0:
        call = lambda *a: L.orc_paged_decode_attention(*a)           # noqa: E731
    elif window == 0:
        call = lambda B_, H_, *a: L.orc_paged_decode_attention_gqa(B_, H_, group, *a)  # noqa: E731
    else:
        call = lambda B_, H_, *a: L.orc_paged_decode_attention_ex(B_, H_, group, window,  # noqa
                                                                  *a)
    rc = call(
        B, H, D, P, dtype, k_pool.ctypes.data, v_pool.ctypes.data, n_pages, q.ctypes.data,
        k_new.ctypes.data, v_new.ctypes.data, tables.ctypes.data, tables.shape[1],
        seq_lens.ctypes.data, out.ctypes.data,
        lane_arr.ctypes.data if lane_arr is not None else None, n_lanes, threads)
    if rc != 0:
        raise ValueError("oracle: sequence length or page id out of range")
    return out


def paged_prefill(k_pool: np.ndarray, v_pool: np.ndarray, q: np.ndarray, k_new: np.ndarray,
                  v_new: np.ndarray, cu_new: np.ndarray, tables: np.ndarray, seq_lens: np.ndarray,
                  dtype: int = F32, group: int = 1, window: int = 0, threads: int = 0,
                  library=None) -> np.ndarray:
    """Chunked prefill: request b appends cu_new[b+1]-cu_new[b] tokens after its
    seq_lens[b] - n_b cached ones; each new token attends causally.  q [N, H*group, D]
    fp32, k_new / v_new [N, H, D] storage dtype, N = cu_new[-1].  Pools are modified in
    place.  Returns out [N, H*group, D] fp64."""
    _check_pool(k_pool, dtype)
    _check_pool(v_pool, dtype)
    n_pages, H, P, D = k_pool.shape
    cu_new = np.ascontiguousarray(cu_new, dtype=np.int32)
    B = cu_new.size - 1
    N = int(cu_new[-1])
    q = np.ascontiguousarray(q, dtype=np.float32)
    assert q.shape == (N, H * group, D)
    k_new = np.ascontiguousarray(k_new, dtype=_storage_dtype(dtype))
    v_new = np.ascontiguousarray(v_new, dtype=_storage_dtype(dtype))
    assert k_new.shape == (N, H, D) and v_new.shape == (N, H, D)
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    assert tables.shape[0] == B and seq_lens.shape == (B,)
    out = np.zeros((N, H * group, D), dtype=np.float64)
    rc = (library or lib()).orc_paged_prefill(
        B, H, group, window, D, P, dtype, k_pool.ctypes.data, v_pool.ctypes.data, n_pages,
        q.ctypes.data, k_new.ctypes.data, v_new.ctypes.data, cu_new.ctypes.data,
        tables.ctypes.data, tables.shape[1], seq_lens.ctypes.data, out.ctypes.data, threads)
    if rc != 0:
        raise ValueError("oracle: sequence length or page id out of range")
    return out


def append(k_pool: np.ndarray, v_pool: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
           tables: np.ndarray, seq_lens: np.ndarray, dtype: int = F32) -> None:
    """Only the append step: write the new rows into slot t_b - 1."""
    _check_pool(k_pool, dtype)
    _check_pool(v_pool, dtype)
    n_pages, H, P, D = k_pool.shape
    B = seq_lens.shape[0]
    k_new = np.ascontiguousarray(k_new, dtype=_storage_dtype(dtype))
    v_new = np.ascontiguousarray(v_new, dtype=_storage_dtype(dtype))
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    rc = lib().orc_append(B, H, D, P, dtype, k_pool.ctypes.data, v_pool.ctypes.data, n_pages,
                          k_new.ctypes.data, v_new.ctypes.data, tables.ctypes.data,
                          tables.shape[1], seq_lens.ctypes.data)
    if rc != 0:
        raise ValueError("oracle: sequence length or page id out of range")


def max_threads() -> int:
    return int(lib().orc_max_threads())


from .model import (  # noqa: E402
    Status, OraclePool, OracleRequest, OracleError, cached_score_cells,
)

__all__ = ["F32", "BF16", "build", "paged_decode_attention", "paged_prefill", "append",
           "max_threads", "Status",
           "OraclePool", "OracleRequest", "OracleError", "cached_score_cells"]
