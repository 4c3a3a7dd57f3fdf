"""The C-ABI library builds, loads without a GPU and exports every declared entry point."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvinc.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("kv_cache_create", "kv_cache_destroy", "kv_reset", "kv_append",
                     "kv_advance", "kv_nbytes", "kv_get_lens", "kv_debug_ptrs", "kv_strerror"):
        assert required in names


def test_library_exports_every_declared_symbol():
    from kv_cache_incremental_gb300 import _build
    lib = ctypes.CDLL(_build.build())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_signatures_cover_the_header():
    from kv_cache_incremental_gb300 import _lib
    assert sorted(_lib.SIGNATURES) == declared_functions()


def test_strerror_and_null_handling_need_no_gpu():
    from kv_cache_incremental_gb300 import _lib
    lib = _lib.load()
    assert lib.kv_strerror(0) == b"KV_OK"
    assert b"full" in lib.kv_strerror(2)
    assert lib.kv_nbytes(None) == -1
    assert lib.kv_append(None, 0, None, None, None, 4, 1, None, None, 0, None, None) == 1
    assert lib.kv_advance(None, None, None, 0, None) == 1
    out = ctypes.c_void_p(123)
    kinds = (ctypes.c_int32 * 1)(0)
    # invalid shapes are rejected before any CUDA call, and *out is cleared
    assert lib.kv_cache_create(ctypes.byref(out), 2, 16, 3, 2, 64, 0, 1, kinds, 1e4, 0) == 1
    assert out.value is None
    assert lib.kv_cache_create(ctypes.byref(out), 2, 16, 4, 2, 96, 0, 1, kinds, 1e4, 0) == 1
    assert lib.kv_cache_create(ctypes.byref(out), 2, 16, 4, 2, 64, 0, 1, kinds, -1.0, 0) == 1
    sliding = (ctypes.c_int32 * 1)(1)
    assert lib.kv_cache_create(ctypes.byref(out), 2, 16, 4, 2, 64, 0, 1, sliding, 1e4, 0) == 1
    assert lib.kv_cache_create(ctypes.byref(out), 2, 16, 64, 2, 64, 0, 1, kinds, 1e4, 0) == 1
    # a paged cache needs a pool; *out is cleared on that refusal too
    out.value = 123
    assert lib.kv_cache_create_paged(ctypes.byref(out), 2, 16, 4, 2, 64, 0, 1, kinds, 1e4, 0,
                                     0) == 1
    assert out.value is None
    # ring rows beyond TMA's 2^31 row coordinates (65536 rows x 16 heads x 2049 slots), on
    # a paged cache whose global pool is small: refused before any CUDA call
    assert lib.kv_cache_create_paged(ctypes.byref(out), 65536, 4096, 16, 16, 64, 2048, 1,
                                     sliding, 1e4, 0, 1) == 1
    # a refused step graph leaves *out NULL
    g = ctypes.c_void_p(77)
    assert lib.kv_step_graph_create(None, ctypes.byref(g), None, None, None, None, 4, None,
                                    1) == 1
    assert g.value is None


def test_package_import_fails_loudly_without_library(tmp_path, monkeypatch):
    from kv_cache_incremental_gb300 import _build, _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib.load(build_if_missing=False)
