"""Python binding of libkvinc: a preallocated per-row KV cache for incremental decoding
on one GB300.

Argument marshalling only: every step of the path (RoPE, append, attention, ring
commit, state updates) runs in the library's CUDA kernels.  PyTorch provides device
memory and streams.  Importing this package loads ``libkvinc.so`` (building it
in-tree when absent) and raises if that fails -- there is no CPU fallback.

    cache = KVCache(B=64, max_len=8192, Hq=32, Hk=8, D=128)
    out = cache.append(0, q, k, v, n_new)     # per layer; does not advance
    cache.advance(n_new)                      # once per step, after all layers
"""
from __future__ import annotations

import ctypes
import weakref
from typing import Optional, Sequence

import numpy as np

from ._lib import (KERNELS, KV_GLOBAL, KV_HYBRID_FULL, KV_HYBRID_LOCAL, KV_SLIDING, KVCacheFull,
                   KVError, KVPoolExhausted, check, load)

__all__ = ["KVCache", "StepGraph", "KVError", "KVCacheFull", "KVPoolExhausted", "KV_GLOBAL",
           "KV_SLIDING", "KV_HYBRID_FULL", "KV_HYBRID_LOCAL", "load", "plan_decode",
           "plan_prefill"]

_clib = load()


_P_I32 = ctypes.POINTER(ctypes.c_int32)


def _i32_array(values):
    """Host int32 array for the C ABI: a pointer into a numpy buffer it keeps alive (values
    that do not fit int32 raise OverflowError)."""
    if values is None:
        return None
    a = np.ascontiguousarray(values, dtype=np.int32).reshape(-1)
    if a.size == 0:
        a = np.zeros(1, dtype=np.int32)
    return a.ctypes.data_as(_P_I32)


class _I32Memo:
    """The last list marshalled for one argument and its int32 array: decode loops pass the
    same per-row counts every step (e.g. [1] * B), which then cost a list comparison instead
    of a conversion."""

    __slots__ = ("key", "ptr")

    def __init__(self):
        self.key, self.ptr = None, None

    def get(self, values):
        if values is None:
            return None
        if type(values) is list and values == self.key:
            return self.ptr
        ptr = _i32_array(values)
        if type(values) is list:
            self.key, self.ptr = list(values), ptr
        return ptr


def _stream_ptr(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


class _DevArray:
    """Zero-copy __cuda_array_interface__ view of library-owned device memory."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


class KVCache:
    """A cache of B rows; see include/kvinc.h for the full contract."""

    def __init__(self, B: int, max_len: int, Hq: int, Hk: int, D: int, W: int = 0,
                 layer_kinds: Sequence[int] = (KV_GLOBAL,), rope_theta: float = 1e4,
                 device: int = 0, paged_blocks: Optional[int] = None):
        """paged_blocks: global layers in a pool of that many 16-position blocks
        (kv_cache_create_paged) instead of max_len slots per row."""
        kinds = _i32_array(layer_kinds)
        h = ctypes.c_void_p()
        if paged_blocks is None:
            check(_clib.kv_cache_create(ctypes.byref(h), B, max_len, Hq, Hk, D, W,
                                       len(layer_kinds), kinds, float(rope_theta), device),
                  "kv_cache_create")
        else:
            check(_clib.kv_cache_create_paged(ctypes.byref(h), B, max_len, Hq, Hk, D, W,
                                             len(layer_kinds), kinds, float(rope_theta), device,
                                             int(paged_blocks)), "kv_cache_create_paged")
        self.paged_blocks = paged_blocks
        self._h = h
        self.B, self.max_len, self.Hq, self.Hk, self.D, self.W = B, max_len, Hq, Hk, D, W
        self.layer_kinds = list(layer_kinds)
        self.device = device
        r = ctypes.c_int()
        _clib.kv_get_config(h, None, None, None, None, None, None, ctypes.byref(r), None)
        self.R = r.value
        self._graphs = weakref.WeakSet()  # step graphs over this cache, closed before it
        self._memo_n, self._memo_rows = _I32Memo(), _I32Memo()

    # ------------------------------------------------------------------ lifecycle
    def close(self) -> None:
        for g in list(getattr(self, "_graphs", ())):
            g.close()
        if getattr(self, "_h", None):
            _clib.kv_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ checks
    def _check_tensor(self, x, name, heads, C=None, Bs=None):
        import torch
        if x.dtype != torch.bfloat16:
            raise TypeError(f"{name}: cache dtype bfloat16 != incoming dtype {x.dtype}")
        if not x.is_cuda or x.device.index != self.device:
            raise ValueError(f"{name} must live on cuda:{self.device}")
        if x.dim() != 4 or x.shape[2] != heads or x.shape[3] != self.D:
            raise ValueError(f"{name}: expected (Bs, C, {heads}, {self.D}), got {tuple(x.shape)}")
        if C is not None and (x.shape[1] != C or x.shape[0] != Bs):
            raise ValueError(f"{name}: shape {tuple(x.shape)} does not match q")
        if not x.is_contiguous():
            raise ValueError(f"{name} must be contiguous")

    # ------------------------------------------------------------------ the path
    def append(self, layer: int, q, k, v, n_new, rows=None, out=None, stream=None):
        """Rotate, append and attend one layer's right-padded chunk; returns out (Bs,C,Hq,D)."""
        import torch
        self._check_tensor(q, "q", self.Hq)
        Bs, C = q.shape[0], q.shape[1]
        self._check_tensor(k, "k", self.Hk, C, Bs)
        self._check_tensor(v, "v", self.Hk, C, Bs)
        if out is None:
            out = torch.empty_like(q)
        else:
            self._check_tensor(out, "out", self.Hq, C, Bs)
        if len(n_new) != Bs or (rows is not None and len(rows) != Bs):
            raise ValueError("n_new and rows must have one entry per row of q")
        check(_clib.kv_append(self._h, layer, q.data_ptr(), k.data_ptr(), v.data_ptr(), self.Hq, C,
                             self._memo_n.get(n_new), self._memo_rows.get(rows), Bs,
                             out.data_ptr(), _stream_ptr(stream, q.device)), "kv_append")
        return out

    def append_hybrid(self, layer: int, q, k_local, v_local, n_new, k_global=None,
                      v_global=None, rows=None, out=None, stream=None):
        """append() for a hybrid layer: k_local, v_local go to the layer's ring; k_global,
        v_global (a KV_HYBRID_FULL layer only) to its group's cache.  One softmax over the
        group's global keys <= p and the layer's local keys in the window."""
        import torch
        self._check_tensor(q, "q", self.Hq)
        Bs, C = q.shape[0], q.shape[1]
        for x, name in ((k_local, "k_local"), (v_local, "v_local"), (k_global, "k_global"),
                        (v_global, "v_global")):
            if x is not None:
                self._check_tensor(x, name, self.Hk, C, Bs)
        if out is None:
            out = torch.empty_like(q)
        else:
            self._check_tensor(out, "out", self.Hq, C, Bs)
        if len(n_new) != Bs or (rows is not None and len(rows) != Bs):
            raise ValueError("n_new and rows must have one entry per row of q")
        ptr = lambda x: None if x is None else x.data_ptr()
        check(_clib.kv_append_hybrid(self._h, layer, q.data_ptr(), k_local.data_ptr(),
                                    v_local.data_ptr(), ptr(k_global), ptr(v_global), self.Hq,
                                    C, _i32_array(n_new), _i32_array(rows), Bs, out.data_ptr(),
                                    _stream_ptr(stream, q.device)), "kv_append_hybrid")
        return out

    def ring_storage(self, layer: int):
        """Zero-copy torch views (K, V) of a hybrid layer's ring, [B, Hk, R + 1, D] bf16."""
        import torch
        kp, vp = ctypes.c_void_p(), ctypes.c_void_p()
        check(_clib.kv_debug_ring_ptrs(self._h, layer, ctypes.byref(kp), ctypes.byref(vp)))
        dev = f"cuda:{self.device}"
        shape = (self.B, self.Hk, self.R + 1, self.D)
        K = torch.as_tensor(_DevArray(kp.value, shape, "<i2"), device=dev).view(torch.bfloat16)
        V = torch.as_tensor(_DevArray(vp.value, shape, "<i2"), device=dev).view(torch.bfloat16)
        return K, V

    def copy_rows(self, src: "KVCache", src_rows, dst_rows, keep=None, stream=None) -> None:
        """Rows dst_rows of this cache become the first keep[i] tokens (default: all) of
        rows src_rows of `src` (this cache or another of the same layout)."""
        import torch
        n = len(src_rows)
        if len(dst_rows) != n or (keep is not None and len(keep) != n):
            raise ValueError("src_rows, dst_rows and keep need one entry per copy")
        check(_clib.kv_copy_rows(self._h, _i32_array(dst_rows), src._h, _i32_array(src_rows),
                                _i32_array(keep), n,
                                _stream_ptr(stream, torch.device("cuda", self.device))),
              "kv_copy_rows")

    def export_row(self, row: int, keep: Optional[int] = None, stream=None):
        """The first `keep` tokens (default: all) of a row as a flat uint8 device tensor."""
        import torch
        keep = self.lens[row] if keep is None else keep
        nbytes = _clib.kv_export_bytes(self._h, keep)
        if nbytes < 0:
            raise ValueError(f"keep={keep} out of range")
        buf = torch.empty(max(16, nbytes), dtype=torch.uint8, device=f"cuda:{self.device}")
        check(_clib.kv_export_row(self._h, row, keep, buf.data_ptr(), nbytes,
                                 _stream_ptr(stream, buf.device)), "kv_export_row")
        return buf[:nbytes]

    def import_row(self, row: int, buf, keep: int, stream=None) -> None:
        """Make `row` the state exported as `buf` (a tensor from export_row) at length keep."""
        if not buf.is_cuda or buf.device.index != self.device:
            raise ValueError(f"buf must live on cuda:{self.device}")
        check(_clib.kv_import_row(self._h, row, keep, buf.data_ptr(), buf.numel() *
                                 buf.element_size(), _stream_ptr(stream, buf.device)),
              "kv_import_row")

    def step_graph(self, q, k, v, out, rows=None, k_global=None, v_global=None) -> "StepGraph":
        """A static-shape decode step (every layer, one token per row, then advance) as a
        CUDA graph over fixed per-layer buffers q[l], k[l], v[l], out[l] of shape
        (Bs, 1, heads, D); hybrid full layers also take k_global[l], v_global[l]; see
        StepGraph."""
        return StepGraph(self, q, k, v, out, rows, k_global, v_global)

    def append_host(self, layer: int, q, k, v, n_new, rows=None, out=None, stream=None):
        """append() for CPU tensors (pinned for asynchronous copies); synchronise the stream
        before reading `out`."""
        import torch
        for x, name in ((q, "q"), (k, "k"), (v, "v")):
            if x.dtype != torch.bfloat16:
                raise TypeError(f"{name}: cache dtype bfloat16 != incoming dtype {x.dtype}")
            if x.is_cuda or not x.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CPU tensor")
        Bs, C = q.shape[0], q.shape[1]
        if out is None:
            out = torch.empty_like(q)
        check(_clib.kv_append_host(self._h, layer, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                  self.Hq, C, _i32_array(n_new), _i32_array(rows), Bs,
                                  out.data_ptr(), _stream_ptr(stream, self.device)),
              "kv_append_host")
        return out

    def append_hybrid_host(self, layer: int, q, k_local, v_local, n_new, k_global=None,
                           v_global=None, rows=None, out=None, stream=None):
        """append_hybrid() for CPU tensors (pinned for asynchronous copies); synchronise the
        stream before reading `out`."""
        import torch
        for x, name in ((q, "q"), (k_local, "k_local"), (v_local, "v_local"),
                        (k_global, "k_global"), (v_global, "v_global")):
            if x is None:
                continue
            if x.dtype != torch.bfloat16:
                raise TypeError(f"{name}: cache dtype bfloat16 != incoming dtype {x.dtype}")
            if x.is_cuda or not x.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CPU tensor")
        Bs, C = q.shape[0], q.shape[1]
        if out is None:
            out = torch.empty_like(q)
        ptr = lambda x: None if x is None else x.data_ptr()
        check(_clib.kv_append_hybrid_host(self._h, layer, q.data_ptr(), k_local.data_ptr(),
                                         v_local.data_ptr(), ptr(k_global), ptr(v_global),
                                         self.Hq, C, _i32_array(n_new), _i32_array(rows), Bs,
                                         out.data_ptr(), _stream_ptr(stream, self.device)),
              "kv_append_hybrid_host")
        return out

    def advance(self, n_new, rows=None, stream=None) -> None:
        """End the step: lens[row] += n_new (call once, after every layer was appended)."""
        Bs = len(n_new)
        check(_clib.kv_advance(self._h, self._memo_n.get(n_new), self._memo_rows.get(rows), Bs,
                              _stream_ptr(stream, self.device)), "kv_advance")

    def reset(self, rows, stream=None) -> None:
        rows = list(rows)
        check(_clib.kv_reset(self._h, _i32_array(rows), len(rows),
                            _stream_ptr(stream, self.device)), "kv_reset")

    # ------------------------------------------------------------------ inspection
    @property
    def lens(self):
        arr = (ctypes.c_int32 * self.B)()
        check(_clib.kv_get_lens(self._h, arr))
        return list(arr)

    def nbytes(self) -> int:
        return int(_clib.kv_nbytes(self._h))

    def storage(self, layer: int):
        """Torch views (K, V) of a layer's storage, [B, Hk, rows, D] bf16; rows = max_len + 1
        (global, and a hybrid layer's group cache) or R + 1 (sliding).  Zero-copy and valid
        while the cache lives, except for a paged cache's global layers: there each row's
        blocks are gathered from the pool into a new tensor (slots past the row's blocks are
        zero)."""
        import torch
        kp, vp, lp = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
        check(_clib.kv_debug_ptrs(self._h, layer, ctypes.byref(kp), ctypes.byref(vp),
                                 ctypes.byref(lp)))
        dev = f"cuda:{self.device}"
        if self.paged_blocks is not None and self.layer_kinds[layer] != KV_SLIDING:
            pool = (self.Hk, self.paged_blocks, 16, self.D)   # head-major pool
            Kp = torch.as_tensor(_DevArray(kp.value, pool, "<i2"), device=dev).view(torch.bfloat16)
            Vp = torch.as_tensor(_DevArray(vp.value, pool, "<i2"), device=dev).view(torch.bfloat16)
            Kp, Vp = Kp.transpose(0, 1), Vp.transpose(0, 1)  # [block][Hk][16][D]
            shape = (self.B, self.Hk, self.max_len + 1, self.D)
            K = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
            V = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
            for b in range(self.B):
                blocks = self.block_table(b)
                if blocks:
                    idx = torch.tensor(blocks, device=dev)
                    n = 16 * len(blocks)
                    m = min(n, self.max_len + 1)
                    K[b, :, :m] = Kp[idx].permute(1, 0, 2, 3).reshape(self.Hk, n, self.D)[:, :m]
                    V[b, :, :m] = Vp[idx].permute(1, 0, 2, 3).reshape(self.Hk, n, self.D)[:, :m]
            return K, V
        rows = self.R + 1 if self.layer_kinds[layer] == KV_SLIDING else self.max_len + 1
        shape = (self.B, self.Hk, rows, self.D)
        K = torch.as_tensor(_DevArray(kp.value, shape, "<i2"), device=dev).view(torch.bfloat16)
        V = torch.as_tensor(_DevArray(vp.value, shape, "<i2"), device=dev).view(torch.bfloat16)
        return K, V

    def block_table(self, row: int):
        """Pool blocks of a row in position order (paged caches; [] otherwise)."""
        n = ctypes.c_int()
        check(_clib.kv_get_block_table(self._h, row, None, 0, ctypes.byref(n)))
        buf = (ctypes.c_int32 * max(1, n.value))()
        check(_clib.kv_get_block_table(self._h, row, buf, n.value, ctypes.byref(n)))
        return list(buf[:n.value])

    @property
    def free_blocks(self) -> int:
        return _clib.kv_free_blocks(self._h)

    def lpos(self):
        """Zero-copy view of lpos [B, R] int32 (position held by each ring slot, -1 empty)."""
        import torch
        lp = ctypes.c_void_p()
        check(_clib.kv_debug_ptrs(self._h, 0, None, None, ctypes.byref(lp)))
        if not lp.value:
            return None
        return torch.as_tensor(_DevArray(lp.value, (self.B, self.R), "<i4"),
                               device=f"cuda:{self.device}")

    def debug_wait_timeout(self, limit: int = 4096, stream=None) -> None:
        """Enqueue a kernel whose bounded wait runs out (kv_debug_wait_timeout); the timeout
        then shows in device_error()."""
        check(_clib.kv_debug_wait_timeout(self._h, int(limit), _stream_ptr(stream, self.device)),
              "kv_debug_wait_timeout")

    def device_error(self) -> int:
        code = ctypes.c_int32()
        _clib.kv_device_error(self._h, ctypes.byref(code))
        return code.value

    # ------------------------------------------------------------------ profiling
    def profile(self, enable: bool = True) -> None:
        check(_clib.kv_profile_enable(self._h, 1 if enable else 0))

    def profile_read(self, kernel: str, reset: bool = False) -> dict:
        n, ms, by, fl = ctypes.c_int64(), ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
        check(_clib.kv_profile_read(self._h, KERNELS[kernel], 1 if reset else 0, ctypes.byref(n),
                                   ctypes.byref(ms), ctypes.byref(by), ctypes.byref(fl)))
        return {"launches": n.value, "ms": ms.value, "bytes": by.value, "flops": fl.value}


class StepGraph:
    """One decode step of a fixed row set, replayed as a CUDA graph (kv_step_graph_*).

    ``launch()`` is equivalent to ``cache.append(l, q[l], k[l], v[l], [1] * Bs, rows,
    out=out[l])`` for every layer followed by ``cache.advance([1] * Bs, rows)``: write the
    step's inputs into the buffers given at construction, then launch.  On a cache with
    hybrid layers, k[l], v[l] of a hybrid layer are its local keys and values and
    k_global[l], v_global[l] the group's global ones (given for KV_HYBRID_FULL layers,
    None elsewhere), as in append_hybrid.  The buffers must stay alive as long as the graph.
    """

    def __init__(self, cache: KVCache, q, k, v, out, rows=None, k_global=None, v_global=None):
        Bs = q[0].shape[0] if len(q) else 0
        self.hybrid = any(kind in (KV_HYBRID_FULL, KV_HYBRID_LOCAL) for kind in cache.layer_kinds)
        self._check(cache, q, k, v, out, Bs, k_global, v_global)
        if rows is not None and len(rows) != Bs:
            raise ValueError("rows must have one entry per row of q")
        h = ctypes.c_void_p()
        if self.hybrid:
            qp, kp, vp, op = self._ptrs(q, k, v, out)
            gk, gv = self._ptrs(self._opt(k_global, len(q)), self._opt(v_global, len(q)))
            check(_clib.kv_step_graph_create_hybrid(cache._h, ctypes.byref(h), qp, kp, vp, gk, gv,
                                                   op, cache.Hq, _i32_array(rows), Bs),
                  "kv_step_graph_create_hybrid")
        else:
            check(_clib.kv_step_graph_create(cache._h, ctypes.byref(h),
                                            *self._ptrs(q, k, v, out), cache.Hq,
                                            _i32_array(rows), Bs), "kv_step_graph_create")
        self._h, self.cache, self.Bs = h, cache, Bs
        # the graph reads these buffers
        self._keep = (list(q), list(k), list(v), list(out), k_global, v_global)
        cache._graphs.add(self)

    @staticmethod
    def _opt(ts, n):
        return [None] * n if ts is None else list(ts)

    @staticmethod
    def _check(cache, q, k, v, out, Bs, k_global=None, v_global=None):
        n = len(cache.layer_kinds)
        if not (len(q) == len(k) == len(v) == len(out) == n):
            raise ValueError(f"one q, k, v and out tensor per layer ({n})")
        for l in range(n):
            cache._check_tensor(q[l], f"q[{l}]", cache.Hq, 1, Bs)
            cache._check_tensor(k[l], f"k[{l}]", cache.Hk, 1, Bs)
            cache._check_tensor(v[l], f"v[{l}]", cache.Hk, 1, Bs)
            cache._check_tensor(out[l], f"out[{l}]", cache.Hq, 1, Bs)
        for name, ts in (("k_global", k_global), ("v_global", v_global)):
            ts = StepGraph._opt(ts, n)
            if len(ts) != n:
                raise ValueError(f"{name}: one entry per layer ({n})")
            for l, t in enumerate(ts):
                if (t is not None) != (cache.layer_kinds[l] == KV_HYBRID_FULL):
                    raise ValueError(f"{name}[{l}]: a tensor exactly on KV_HYBRID_FULL layers")
                if t is not None:
                    cache._check_tensor(t, f"{name}[{l}]", cache.Hk, 1, Bs)
        return Bs

    @staticmethod
    def _ptrs(*groups):
        return [(ctypes.c_void_p * len(ts))(*[None if t is None else t.data_ptr() for t in ts])
                for ts in groups]

    def buffers(self, q, k, v, out, k_global=None, v_global=None) -> "StepBuffers":
        """A validated set of per-layer buffers (same shapes as at construction) that
        launch(buffers=...) switches to without further checks."""
        self._check(self.cache, q, k, v, out, self.Bs, k_global, v_global)
        n = len(q)
        ptrs = self._ptrs(q, k, v, self._opt(k_global, n), self._opt(v_global, n), out)
        return StepBuffers(ptrs, (list(q), list(k), list(v), list(out), k_global, v_global))

    def set_buffers(self, q, k, v, out, k_global=None, v_global=None) -> None:
        """Point the following launches at other per-layer buffers of the same shapes."""
        self._use(self.buffers(q, k, v, out, k_global, v_global))

    def _use(self, b: "StepBuffers") -> None:
        qp, kp, vp, gk, gv, op = b.ptrs
        if self.hybrid:
            check(_clib.kv_step_graph_set_buffers_hybrid(self._h, qp, kp, vp, gk, gv, op),
                  "kv_step_graph_set_buffers_hybrid")
        else:
            check(_clib.kv_step_graph_set_buffers(self._h, qp, kp, vp, op),
                  "kv_step_graph_set_buffers")
        self._keep = b.tensors

    def launch(self, stream=None, buffers: Optional["StepBuffers"] = None) -> None:
        """One decode step of every layer, then advance; with `buffers`, this step (and the
        following ones) read and write that buffer set."""
        import torch
        if buffers is not None:
            self._use(buffers)
        check(_clib.kv_step_graph_launch(self._h, _stream_ptr(stream, torch.device(
            "cuda", self.cache.device))), "kv_step_graph_launch")

    def close(self) -> None:
        if getattr(self, "_h", None):
            _clib.kv_step_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class StepBuffers:
    """Per-layer q, k, v, out buffers checked once for a StepGraph (see StepGraph.buffers)."""

    def __init__(self, ptrs, tensors):
        self.ptrs, self.tensors = ptrs, tensors


def plan_decode(num_sms: int, Hq: int, Hk: int, D: int, R: int, kind: int, pos) -> dict:
    """The split-K schedule of one decode launch (kv_plan_decode): per row the splits and
    64-key tiles per split of its storage segment and of a hybrid layer's ring, its first
    partial slot (-1: one split, no merge), and the launch's CTAs per kv head.  Host only."""
    n = len(pos)
    outs = [(ctypes.c_int32 * max(1, n))() for _ in range(5)]
    items = ctypes.c_int32()
    check(_clib.kv_plan_decode(num_sms, Hq, Hk, D, R, kind, n, _i32_array(pos), *outs,
                               ctypes.byref(items)), "kv_plan_decode")
    names = ("n_splits", "split_tiles", "n_splits2", "split_tiles2", "part0")
    plan = {k: list(a)[:n] for k, a in zip(names, outs)}
    plan["n_items"] = items.value
    return plan


def plan_prefill(num_sms: int, Hq: int, Hk: int, D: int, R: int, kind: int, lens, n) -> dict:
    """The prefill launches of one sub-chunk (kv_plan_prefill): the entries in launch order
    (input row, kernel kind, 64-key tile range, first partial vector or -1), the entries
    per row and the partial vectors.  Host only."""
    rows = len(lens)
    if len(n) != rows:
        raise ValueError("lens and n differ in length")
    count, vecs = ctypes.c_int32(), ctypes.c_int64()
    splits = (ctypes.c_int32 * max(1, rows))()
    args = (num_sms, Hq, Hk, D, R, kind, rows, _i32_array(lens), _i32_array(n))
    _clib.kv_plan_prefill(*args, 0, None, None, None, None, None, ctypes.byref(count), splits,
                          ctypes.byref(vecs))
    cap = count.value
    ents = [(ctypes.c_int32 * max(1, cap))() for _ in range(5)]
    check(_clib.kv_plan_prefill(*args, cap, *ents, ctypes.byref(count), splits,
                                ctypes.byref(vecs)), "kv_plan_prefill")
    names = ("row", "kind", "tile0", "tile1", "part")
    plan = {k: list(a)[:cap] for k, a in zip(names, ents)}
    plan["n_splits"] = list(splits)[:rows]
    plan["part_vecs"] = vecs.value
    return plan
