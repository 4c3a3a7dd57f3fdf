"""ctypes loader for libkvinc.so: signatures of every entry point of include/kvinc.h.

There is no fallback: if the shared library is missing or fails to load, importing
the binding raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

c_int, c_int32, c_int64, c_double, c_void_p = (ctypes.c_int, ctypes.c_int32, ctypes.c_int64,
                                               ctypes.c_double, ctypes.c_void_p)
P_i32 = ctypes.POINTER(ctypes.c_int32)

KV_GLOBAL, KV_SLIDING, KV_HYBRID_FULL, KV_HYBRID_LOCAL = 0, 1, 2, 3
(KV_OK, KV_ERR_ARG, KV_ERR_FULL, KV_ERR_DTYPE, KV_ERR_CUDA, KV_ERR_OOM, KV_ERR_DEVICE,
 KV_ERR_SCRATCH, KV_ERR_POOL) = range(9)
KERNELS = {"append": 0, "decode": 1, "combine": 2, "prefill": 3, "commit": 4, "state": 5,
           "step": 6}

# name -> (restype, argtypes); mirrors include/kvinc.h
SIGNATURES = {
    "kv_cache_create": (c_int, [ctypes.POINTER(c_void_p), c_int, c_int, c_int, c_int, c_int, c_int,
                                c_int, P_i32, c_double, c_int]),
    "kv_cache_create_paged": (c_int, [ctypes.POINTER(c_void_p), c_int, c_int, c_int, c_int, c_int,
                                      c_int, c_int, P_i32, c_double, c_int, c_int]),
    "kv_get_block_table": (c_int, [c_void_p, c_int, P_i32, c_int, ctypes.POINTER(c_int)]),
    "kv_free_blocks": (c_int, [c_void_p]),
    "kv_cache_destroy": (None, [c_void_p]),
    "kv_reset": (c_int, [c_void_p, P_i32, c_int, c_void_p]),
    "kv_append": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int, c_int, P_i32, P_i32,
                          c_int, c_void_p, c_void_p]),
    "kv_append_hybrid": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_int, c_int, P_i32, P_i32, c_int, c_void_p, c_void_p]),
    "kv_append_hybrid_host": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_int, c_int, P_i32, P_i32, c_int, c_void_p,
                                      c_void_p]),
    "kv_append_host": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int, c_int, P_i32,
                               P_i32, c_int, c_void_p, c_void_p]),
    "kv_advance": (c_int, [c_void_p, P_i32, P_i32, c_int, c_void_p]),
    "kv_nbytes": (c_int64, [c_void_p]),
    "kv_get_lens": (c_int, [c_void_p, P_i32]),
    "kv_debug_ptrs": (c_int, [c_void_p, c_int, ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p),
                              ctypes.POINTER(c_void_p)]),
    "kv_debug_ring_ptrs": (c_int, [c_void_p, c_int, ctypes.POINTER(c_void_p),
                                   ctypes.POINTER(c_void_p)]),
    "kv_get_config": (c_int, [c_void_p] + [ctypes.POINTER(c_int)] * 8),
    "kv_device_error": (c_int, [c_void_p, P_i32]),
    "kv_debug_wait_timeout": (c_int, [c_void_p, ctypes.c_uint32, c_void_p]),
    "kv_plan_decode": (c_int, [c_int] * 7 + [P_i32] * 6 + [P_i32]),
    "kv_plan_prefill": (c_int, [c_int] * 7 + [P_i32, P_i32, c_int] + [P_i32] * 7
                        + [ctypes.POINTER(c_int64)]),
    "kv_profile_enable": (c_int, [c_void_p, c_int]),
    "kv_profile_read": (c_int, [c_void_p, c_int, c_int, ctypes.POINTER(c_int64),
                                ctypes.POINTER(c_double), ctypes.POINTER(c_double),
                                ctypes.POINTER(c_double)]),
    "kv_decode_noalloc": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_void_p,
                                  c_void_p, c_int, P_i32, P_i32, P_i32, c_int, c_void_p,
                                  c_void_p, c_void_p]),
    "kv_step_graph_create": (c_int, [c_void_p, ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p),
                                     ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p),
                                     ctypes.POINTER(c_void_p), c_int, P_i32, c_int]),
    "kv_step_graph_set_buffers": (c_int, [c_void_p, ctypes.POINTER(c_void_p),
                                          ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p),
                                          ctypes.POINTER(c_void_p)]),
    "kv_step_graph_create_hybrid": (c_int, [c_void_p, ctypes.POINTER(c_void_p)]
                                    + [ctypes.POINTER(c_void_p)] * 6 + [c_int, P_i32, c_int]),
    "kv_step_graph_set_buffers_hybrid": (c_int, [c_void_p] + [ctypes.POINTER(c_void_p)] * 6),
    "kv_step_graph_launch": (c_int, [c_void_p, c_void_p]),
    "kv_step_graph_destroy": (None, [c_void_p]),
    "kv_copy_rows": (c_int, [c_void_p, P_i32, c_void_p, P_i32, P_i32, c_int, c_void_p]),
    "kv_export_bytes": (c_int64, [c_void_p, c_int]),
    "kv_export_row": (c_int, [c_void_p, c_int, c_int, c_void_p, c_int64, c_void_p]),
    "kv_import_row": (c_int, [c_void_p, c_int, c_int, c_void_p, c_int64, c_void_p]),
    "kv_strerror": (ctypes.c_char_p, [c_int]),
}

_lib = None


def load(build_if_missing: bool = True):
    """Load libkvinc.so (building it in-tree first when it is absent or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise ImportError(f"libkvinc.so not found at {path}; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class KVError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = load().kv_strerror(code).decode()
        super().__init__(f"{what}: {msg}" if what else msg)


def check(code: int, what: str = "") -> None:
    if code != KV_OK:
        if code == KV_ERR_FULL:
            raise KVCacheFull(code, what)
        if code == KV_ERR_POOL:
            raise KVPoolExhausted(code, what)
        if code == KV_ERR_DTYPE:
            raise TypeError(load().kv_strerror(code).decode())
        raise KVError(code, what)


class KVCacheFull(KVError, ValueError):
    """lens + n_new > max_len for some row (raised before any write)."""


class KVPoolExhausted(KVError):
    """A paged cache has too few free blocks for the call (raised before any write)."""
