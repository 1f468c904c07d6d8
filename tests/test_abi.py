"""The C-ABI library builds, loads, and exports every entry point the header
declares (CPU only: no device work is requested)."""
import ctypes
import os
import re
import subprocess

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "pkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["pkv_pool_create", "pkv_pool_destroy", "pkv_lease_pages", "pkv_release_pages",
                     "pkv_begin_token", "pkv_append_and_attend", "pkv_commit_token",
                     "pkv_abort_token", "pkv_paged_decode_attention", "pkv_workspace_size",
                     "pkv_check_device_status", "pkv_last_error"]:
        assert required in names


def test_library_exports_every_declared_symbol():
    import paged_kv_cache_decode_gb300 as pkv
    lib = ctypes.CDLL(pkv.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # binding covers exactly the declared set
    from paged_kv_cache_decode_gb300.binding import SIGNATURES
    assert sorted(SIGNATURES) == declared_functions()


def test_exported_symbols_are_c_linkage():
    import paged_kv_cache_decode_gb300 as pkv
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b(pkv_[a-z0-9_]+)\b", out))
    assert set(declared_functions()) <= exported


def test_status_strings_and_version():
    import paged_kv_cache_decode_gb300 as pkv
    assert pkv.lib.pkv_version() >= 10000
    assert pkv.lib.pkv_status_string(pkv.PKV_ERR_OUT_OF_PAGES) == b"PKV_ERR_OUT_OF_PAGES"
    assert pkv.lib.pkv_status_string(123) == b"PKV_ERR_UNKNOWN"


def test_missing_library_fails_loudly(tmp_path):
    from paged_kv_cache_decode_gb300 import binding
    with pytest.raises(ImportError):
        binding.load(str(tmp_path / "nope.so"))
