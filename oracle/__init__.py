"""CPU oracle for incremental decoding against a preallocated KV cache.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the product path never
does.  The arithmetic lives in ``oracle.c`` (plain C, double precision for the
attention, float without fused multiply-add for RoPE); this module only builds
it with gcc and marshals numpy arrays through ctypes.

Every function states the passage it follows; the C file lists the readings
taken where the pages leave a step open.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_U16P = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_I32P = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_F32P = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_F64P = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc (OpenMP, no FP contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_rope_table.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, _F32P, _F32P]
        lib.oracle_rope_table.restype = None
        lib.oracle_rope_bf16.argtypes = [_U16P, ctypes.c_int, ctypes.c_int, ctypes.c_double, _U16P]
        lib.oracle_rope_bf16.restype = None
        lib.oracle_rope_rows.argtypes = [_U16P, _I32P, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_double, _U16P]
        lib.oracle_rope_rows.restype = None
        lib.oracle_visible.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_visible.restype = ctypes.c_int
        lib.oracle_ring_positions.argtypes = [ctypes.c_int, ctypes.c_int, _I32P]
        lib.oracle_ring_positions.restype = None
        lib.oracle_attend.argtypes = [_U16P, _I32P, ctypes.c_int, _U16P, _U16P, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_double, _F64P]
        lib.oracle_attend.restype = ctypes.c_int
        lib.oracle_attend_hybrid.argtypes = [_U16P, _I32P, ctypes.c_int, _U16P, _U16P, _U16P,
                                             _U16P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_double, _F64P]
        lib.oracle_attend_hybrid.restype = ctypes.c_int
        lib.oracle_kv_nbytes.argtypes = [ctypes.c_int] * 10
        lib.oracle_kv_nbytes.restype = ctypes.c_int64
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def f32_to_bf16(x) -> np.ndarray:
    """bfloat16 bits of float32 values, round to nearest even (element by element)."""
    lib = _load()
    a = np.asarray(x, dtype=np.float32)
    flat = a.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    for i, f in enumerate(flat):
        out[i] = lib.oracle_f32_to_bf16(float(f))
    return out.reshape(a.shape)


def bf16_to_f32(bits) -> np.ndarray:
    """float32 values of bfloat16 bit patterns (exact widening)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def rope_table(n_pos: int, D: int, theta: float = 1e4):
    """cos/sin tables [n_pos][D/2] as float32.

    Frequencies theta^(-2i/D) over the half-split pairing of
    tiny_agent/generate.py `_rope_pos`; the exponent and angle in double."""
    lib = _load()
    c = np.empty((n_pos, D // 2), dtype=np.float32)
    s = np.empty((n_pos, D // 2), dtype=np.float32)
    lib.oracle_rope_table(n_pos, D, float(theta), c, s)
    return c, s


def rope_bf16(x, positions, theta: float = 1e4) -> np.ndarray:
    """Rotate bf16 head vectors to their absolute positions (tiny_agent/generate.py `_rope_pos`).

    x: uint16 [..., D]; positions: broadcastable to x.shape[:-1]."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    D = x.shape[-1]
    pos = np.ascontiguousarray(
        np.broadcast_to(np.asarray(positions, dtype=np.int32), x.shape[:-1]).reshape(-1))
    flat = np.ascontiguousarray(x.reshape(-1, D))
    out = np.empty_like(flat)
    lib.oracle_rope_rows(flat, pos, flat.shape[0], D, float(theta), out)
    return out.reshape(x.shape)


def visible(p: int, j: int, W: int = 0) -> bool:
    """Offset mask (Lab 07 section 2) with the sliding clamp of the inkling ring-buffer PR."""
    return bool(_load().oracle_visible(int(p), int(j), int(W)))


def ring_positions(lens: int, W: int) -> np.ndarray:
    """Position held by each of the W ring slots after `lens` appended tokens (-1 = empty)."""
    out = np.empty(W, dtype=np.int32)
    _load().oracle_ring_positions(int(lens), int(W), out)
    return out


def attend(q, qpos, k, v, k_base: int, Hq: int, Hk: int, W: int = 0,
           theta: float = 1e4) -> np.ndarray:
    """Cache-free attention of one row's queries over its pre-RoPE key/value history.

    q: uint16 [n_q, Hq, D] (pre-RoPE), qpos: int [n_q] absolute positions,
    k, v: uint16 [n_k, Hk, D] for positions k_base .. k_base+n_k-1.
    Returns float64 [n_q, Hq, D]."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    qpos = np.ascontiguousarray(qpos, dtype=np.int32)
    n_q, hq, D = q.shape
    n_k = k.shape[0]
    assert hq == Hq and k.shape == (n_k, Hk, D) and v.shape == (n_k, Hk, D)
    out = np.zeros((n_q, Hq, D), dtype=np.float64)
    rc = lib.oracle_attend(q, qpos, n_q, k, v, int(k_base), n_k, Hq, Hk, D, int(W),
                           float(theta), out)
    if rc != 0:
        raise ValueError("oracle_attend: invalid arguments or history does not cover the window")
    return out


def attend_hybrid(q, qpos, kg, vg, kl, vl, Hq: int, Hk: int, W: int,
                  theta: float = 1e4) -> np.ndarray:
    """Hybrid attention (tiny_agent/generate.py `_append_chunk`): one softmax over the group's
    global keys at every position <= p and the layer's local keys in its window.

    q: uint16 [n_q, Hq, D] (pre-RoPE), qpos: [n_q]; kg, vg, kl, vl: uint16 [n_k, Hk, D] for
    positions 0 .. n_k-1.  Returns float64 [n_q, Hq, D]."""
    lib = _load()
    arrs = [np.ascontiguousarray(x, dtype=np.uint16) for x in (q, kg, vg, kl, vl)]
    q, kg, vg, kl, vl = arrs
    qpos = np.ascontiguousarray(qpos, dtype=np.int32)
    n_q, hq, D = q.shape
    n_k = kg.shape[0]
    assert hq == Hq and all(x.shape == (n_k, Hk, D) for x in (kg, vg, kl, vl))
    out = np.zeros((n_q, Hq, D), dtype=np.float64)
    rc = lib.oracle_attend_hybrid(q, qpos, n_q, kg, vg, kl, vl, n_k, Hq, Hk, D, int(W),
                                  float(theta), out)
    if rc != 0:
        raise ValueError("oracle_attend_hybrid: invalid arguments or uncovered position")
    return out


def kv_nbytes(B, max_len, W, D, elem_bytes, n_global, Hk_global, n_sliding, Hk_sliding,
              extra_slots) -> int:
    """K+V bytes (Lab 07 "Check yourself" 1; the inkling PR's memory table)."""
    return int(_load().oracle_kv_nbytes(B, max_len, W, D, elem_bytes, n_global, Hk_global,
                                        n_sliding, Hk_sliding, extra_slots))


def num_threads() -> int:
    return int(_load().oracle_num_threads())
