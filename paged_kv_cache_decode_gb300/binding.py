"""ctypes binding of libpkv.so (see include/pkv.h).  Argument marshalling only:
every step of the path runs in the library's kernels.  There is no fallback —
if the library cannot be loaded, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import importlib.util

_spec = importlib.util.spec_from_file_location(
    "_pkv_build", os.path.join(os.path.dirname(os.path.abspath(__file__)), "build.py"))
_build = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(_build)

PKV_OK = 0
PKV_ERR_INVALID_ARGUMENT = 1
PKV_ERR_OUT_OF_PAGES = 2
PKV_ERR_CAPACITY_EXCEEDED = 3
PKV_ERR_BAD_STATE = 4
PKV_ERR_OUT_OF_MEMORY = 5
PKV_ERR_CUDA = 6
PKV_ERR_DEVICE_CHECK = 7
PKV_ERR_NO_STORAGE = 8
PKV_ERR_UNSUPPORTED = 9

PKV_F32 = 0
PKV_BF16 = 1
PKV_POOL_HOST_ONLY = 1
PKV_POOL_CUDA_CORES = 2

PKV_DEVERR_SEQ_LEN = 1
PKV_DEVERR_PAGE_ID = 2
PKV_DEVERR_TIMEOUT = 4
PKV_DEVERR_SHARED = 8

PKV_INJECT_NONE = 0
PKV_INJECT_LEASE = 1
PKV_INJECT_LAYER = 2
PKV_INJECT_DEVICE_WAIT = 3

LIB_PATH = _build.LIB


class pkv_pool_options(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int), ("pages", ctypes.c_int64), ("kv_heads", ctypes.c_int),
                ("query_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("page_size", ctypes.c_int), ("dtype", ctypes.c_int),
                ("max_context", ctypes.c_int64), ("seed", ctypes.c_uint64),
                ("flags", ctypes.c_uint), ("window", ctypes.c_int64)]


class pkv_counters(ctypes.Structure):
    _fields_ = [("committed_tokens", ctypes.c_int64), ("cache_appends", ctypes.c_int64),
                ("score_cells", ctypes.c_int64)]


_i, _i64, _u64, _u32, _vp, _sz = (ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                  ctypes.c_void_p, ctypes.c_size_t)
_P = ctypes.POINTER

# name -> argtypes (restype int unless listed in _RESTYPE)
SIGNATURES = {
    "pkv_pool_create": [_i, _i64, _i, _i, _i, _i, _i64, _u64, ctypes.c_uint, _P(_vp)],
    "pkv_pool_options_init": [_P(pkv_pool_options)],
    "pkv_pool_create_ex": [_P(pkv_pool_options), _P(_vp)],
    "pkv_pool_heads": [_vp, _P(_i), _P(_i)],
    "pkv_pool_kernel": [_vp, _P(_i)],
    "pkv_pool_destroy": [_vp],
    "pkv_pool_kv_ptr": [_vp, _i, _P(_vp), _P(_vp)],
    "pkv_pool_bytes": [_vp, _P(_u64)],
    "pkv_pool_pages": [_vp, _P(_i64), _P(_i64)],
    "pkv_pool_free_list": [_vp, _vp, _i64, _P(_i64)],
    "pkv_request_create": [_vp, _P(_vp)],
    "pkv_request_destroy": [_vp],
    "pkv_request_fork": [_vp, _P(_vp)],
    "pkv_pool_page_refs": [_vp, ctypes.c_int32, _P(_i)],
    "pkv_lease_pages": [_vp, _i64],
    "pkv_release_pages": [_vp],
    "pkv_request_length": [_vp, _P(_i64)],
    "pkv_request_page_table": [_vp, _vp, _i64, _P(_i64)],
    "pkv_request_counters": [_vp, _P(pkv_counters)],
    "pkv_begin_token": [_vp, _P(_i64)],
    "pkv_append_and_attend": [_vp, _i, _vp, _vp, _vp, _vp, _vp],
    "pkv_commit_token": [_vp],
    "pkv_abort_token": [_vp],
    "pkv_workspace_size": [_vp, _i, _i64, _P(_sz)],
    "pkv_paged_decode_attention": [_vp, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _i64, _vp, _vp, _sz,
                                   _vp],
    "pkv_paged_decode_attention_static": [_vp, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _i64, _vp,
                                          _vp],
    "pkv_prefill_workspace_size": [_vp, _i, _i64, _P(_sz)],
    "pkv_paged_prefill": [_vp, _i, _i, _i64, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _sz, _vp],
    "pkv_begin_chunk": [_vp, _i64, _P(_i64)],
    "pkv_prefill_chunk": [_vp, _i, _vp, _vp, _vp, _vp, _vp],
    "pkv_workspace_size_shared": [_vp, _i, _i64, _i64, _P(_sz)],
    "pkv_paged_decode_attention_shared": [_vp, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _i64, _i64,
                                          _vp, _vp, _sz, _vp],
    "pkv_pool_set_timing_events": [_vp, _vp, _vp],
    "pkv_pool_inject_fault": [_vp, _i, _i64, ctypes.c_uint64],
    "pkv_check_device_status": [_vp, _P(_u32)],
    "pkv_last_error": [],
    "pkv_status_string": [_i],
    "pkv_version": [],
}
_RESTYPE = {"pkv_last_error": ctypes.c_char_p, "pkv_status_string": ctypes.c_char_p}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"libpkv.so not found at {path}; build it with "
            "`python paged_kv_cache_decode_gb300/build.py` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, args in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = _RESTYPE.get(name, ctypes.c_int)
    return lib


lib = load()


class PkvError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        msg = lib.pkv_last_error().decode(errors="replace")
        name = lib.pkv_status_string(status).decode()
        super().__init__(f"{call}: {name}: {msg}")


def check(status: int, call: str) -> None:
    if status != PKV_OK:
        raise PkvError(status, call)
