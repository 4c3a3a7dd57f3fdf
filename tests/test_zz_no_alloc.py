"""kv_decode_noalloc: the decode entry point for callers that cannot call cudaMalloc.

Such callers (a process whose device memory belongs to another allocator, or a loop
that must never allocate) pass their own cache storage, queries, RoPE table and
output; the split partials live in the library's fixed device scratch.  These tests
call it through the C ABI and compare it with kv_append, the entry point that uses
memory from kv_cache_create, on two decode calls in a row.  This file is collected
last so that a run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
from harness import Scenario, bf16_bits_to_torch, check_close, torch_to_bits

pytestmark = pytest.mark.gpu


def _i32(vals):
    return (ctypes.c_int32 * len(vals))(*[int(x) for x in vals])


def _rope_table(max_len, D, theta):
    import torch
    c, s = oracle.rope_table(max_len, D, theta)
    tab = np.ascontiguousarray(np.stack([c, s], axis=-1), dtype=np.float32)  # [pos][D/2][2]
    return torch.from_numpy(tab).to("cuda")


def test_noalloc_decode_matches_kv_append_on_two_calls():
    import torch
    from kv_cache_incremental_gb300 import _lib
    lib = _lib.load()
    B, max_len, Hq, Hk, D = 6, 3000, 16, 4, 128
    sc = Scenario(B=B, max_len=max_len, Hq=Hq, Hk=Hk, D=D, seed=21)
    targets = [2900, 700, 65, 1, 1500, 2111]  # many splits, one split, one key
    while any(t > l for t, l in zip(targets, sc.lens)):
        n = [min(64, t - l) for t, l in zip(targets, sc.lens)]
        sc.step(n, C=64, check=False)
    rope = _rope_table(max_len, D, 1e4)
    K, V = sc.cache.storage(0)
    stream = torch.cuda.current_stream().cuda_stream
    rows = list(range(B))
    for call in range(2):
        q, k, v = sc.chunk_inputs(0, rows, [1] * B, 1)
        qt, kt, vt = (bf16_bits_to_torch(x, "cuda") for x in (q, k, v))
        ref = sc.cache.append(0, qt, kt, vt, [1] * B)  # appends the new keys, then attends
        out = torch.full((B, Hq, D), 7.0, dtype=torch.bfloat16, device="cuda")
        pos = list(sc.lens)
        rc = lib.kv_decode_noalloc(K.data_ptr(), V.data_ptr(), B, max_len + 1, Hq, Hk, D,
                                   qt.data_ptr(), rope.data_ptr(), max_len, _i32(rows),
                                   _i32(pos), _i32([p + 1 for p in pos]), B, out.data_ptr(),
                                   ctypes.c_void_p(stream))
        assert rc == 0, lib.kv_strerror(rc)
        torch.cuda.synchronize()
        ref_f = oracle.bf16_to_f32(torch_to_bits(ref)[:, 0]).astype(np.float64)
        check_close(torch_to_bits(out), ref_f, f"call {call}")
        sc.cache.advance([1] * B)
        sc.lens = [l + 1 for l in sc.lens]


def test_noalloc_rejects_requests_beyond_its_scratch():
    import torch
    from kv_cache_incremental_gb300 import _lib
    lib = _lib.load()
    Hq, Hk, D, n_rows = 8, 2, 64, 600
    K = torch.zeros((n_rows, Hk, 4, D), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((n_rows, Hq, D), dtype=torch.bfloat16, device="cuda")
    rope = _rope_table(4, D, 1e4)
    out = torch.zeros_like(q)
    Bs = 513  # one more row than the fixed scratch plans for
    rc = lib.kv_decode_noalloc(K.data_ptr(), K.data_ptr(), n_rows, 4, Hq, Hk, D, q.data_ptr(),
                               rope.data_ptr(), 4, _i32(range(Bs)), _i32([0] * Bs),
                               _i32([1] * Bs), Bs, out.data_ptr(), None)
    assert rc == _lib.KV_ERR_SCRATCH
    assert b"scratch" in lib.kv_strerror(rc)
    assert torch.count_nonzero(out).item() == 0
