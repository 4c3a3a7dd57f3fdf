"""Seeded, counter-based synthetic inputs for the KV-cache workloads.

This module holds none of the attention or cache arithmetic.  It serves both
the CPU oracle (which regenerates any row's history on demand) and the GPU
path (whose large inputs are filled on the device by ``synth_device.cu``,
the same generator written in CUDA).  Both implement one definition:

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) used as a counter-based generator: draw number
  c of a stream with key K is ``mix(K + (c + 1) * GAMMA)``.
* A stream key per (seed, tensor, layer, row, seq), chained through ``mix``.
* Element (pos, head, d) of a tensor with H heads of width D uses counter
  e = (pos * H + head) * D + d and three draws 3e, 3e+1, 3e+2.
* The twelve 16-bit lanes of those draws sum to S; the value is
  (S - 393210) / 65536 in float32 (exact), rounded once to bfloat16.
  This is the Irwin-Hall(12) approximation of N(0, 1): mean 0, variance 1,
  support +-6, computed with integer arithmetic only so that the CPU and
  the GPU produce identical bits.

``tensor`` ids: 0 = q, 1 = k, 2 = v, 3 = a layer group's global k, 4 = its global v (any
other small integer is allowed).
``seq`` counts the sequences a row has held (it changes after a reset).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MEAN12 = 393210  # 12 * 32767.5

Q, K, V, KG, VG = 0, 1, 2, 3, 4


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _mix_int(z: int) -> int:
    m = (1 << 64) - 1
    z &= m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def stream_key(seed: int, tensor: int, layer: int, row: int, seq: int = 0) -> int:
    """64-bit key of one (seed, tensor, layer, row, seq) stream."""
    g = 0x9E3779B97F4A7C15
    m = (1 << 64) - 1
    k = _mix_int((seed + g) & m)
    for x in (tensor, layer, row, seq):
        k = _mix_int((k + (x + 1) * g) & m)
    return k


def _draw(key: int, ctr: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return _mix(np.uint64(key) + (ctr + np.uint64(1)) * GAMMA)


def _lanes_sum(u: np.ndarray) -> np.ndarray:
    s = np.zeros(u.shape, dtype=np.int64)
    for sh in (0, 16, 32, 48):
        s += ((u >> np.uint64(sh)) & np.uint64(0xFFFF)).astype(np.int64)
    return s


def _f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def normal_bf16(seed: int, tensor: int, layer: int, row: int, seq: int,
                positions, H: int, D: int) -> np.ndarray:
    """bf16 bits [len(positions), H, D] of the stream at the given absolute positions."""
    key = stream_key(seed, tensor, layer, row, seq)
    pos = np.asarray(positions, dtype=np.uint64).reshape(-1, 1, 1)
    h = np.arange(H, dtype=np.uint64).reshape(1, -1, 1)
    d = np.arange(D, dtype=np.uint64).reshape(1, 1, -1)
    with np.errstate(over="ignore"):
        e = (pos * np.uint64(H) + h) * np.uint64(D) + d
        s = (_lanes_sum(_draw(key, e * np.uint64(3)))
             + _lanes_sum(_draw(key, e * np.uint64(3) + np.uint64(1)))
             + _lanes_sum(_draw(key, e * np.uint64(3) + np.uint64(2))))
    x = (s - _MEAN12).astype(np.float32) / np.float32(65536.0)
    return _f32_to_bf16_rne(x)


def bf16_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ------------------------------------------------------------------ device side

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_device.cu")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkvsynth.so")
_lock = threading.Lock()
_lib = None


def build_command(out_path: str = _LIB_PATH) -> list:
    return ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
            "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-o", out_path, _SRC]


def build(force: bool = False) -> str:
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(build_command(tmp), check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.kvsynth_fill_bf16.argtypes = [
                ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
            lib.kvsynth_fill_bf16.restype = ctypes.c_int
            _lib = lib
        return _lib


def fill_device(dst_ptr: int, seed: int, tensor: int, layer: int,
                rows_ptr: int, seqs_ptr: int, pos0_ptr: int, n_rows: int,
                C: int, H: int, D: int, stream: int = 0) -> None:
    """Fill a device bf16 tensor [n_rows, C, H, D]: token t of row i is position pos0[i] + t
    of stream (seed, tensor, layer, rows[i], seqs[i]).  rows/seqs/pos0 are device int32
    arrays of length n_rows."""
    rc = _load().kvsynth_fill_bf16(ctypes.c_void_p(dst_ptr), ctypes.c_uint64(seed), tensor,
                                   layer, ctypes.c_void_p(rows_ptr), ctypes.c_void_p(seqs_ptr),
                                   ctypes.c_void_p(pos0_ptr), n_rows, C, H, D,
                                   ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"kvsynth_fill_bf16 failed with CUDA error {rc}")


def fill_torch(out, seed: int, tensor: int, layer: int, rows, seqs, pos0) -> None:
    """Torch convenience: out is a CUDA bf16 tensor [n_rows, C, H, D]; rows/seqs/pos0 are
    sequences of ints (copied to the device here)."""
    import torch
    n, C, H, D = out.shape
    dev = out.device
    meta = torch.tensor([list(rows), list(seqs), list(pos0)], dtype=torch.int32).to(dev)
    fill_device(out.data_ptr(), seed, tensor, layer, meta[0].data_ptr(), meta[1].data_ptr(),
                meta[2].data_ptr(), n, C, H, D, torch.cuda.current_stream(dev).cuda_stream)
