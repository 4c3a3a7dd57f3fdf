"""Host-side error paths of the C ABI on a live cache: every rejected call returns its code
before any work is enqueued and changes no state (pycraft-1 `update` guards; tiny_agent
`append` raises "KV cache full" before writing)."""
import ctypes

import numpy as np
import pytest

from harness import Scenario, torch_to_bits

pytestmark = pytest.mark.gpu


def _i32(v):
    return (ctypes.c_int32 * max(1, len(v)))(*[int(x) for x in v])


@pytest.fixture()
def sc():
    s = Scenario(B=4, max_len=40, Hq=8, Hk=2, D=64, W=8, kinds=[1, 0], seed=17)
    s.step([10, 3, 0, 39], C=39)
    return s


def _snapshot(s):
    import torch
    torch.cuda.synchronize()
    out = [torch_to_bits(x) for layer in range(2) for x in s.cache.storage(layer)]
    out.append(s.cache.lpos().cpu().numpy().copy())
    return out, list(s.cache.lens)


def test_every_rejected_call_changes_nothing(sc):
    import torch
    from kv_cache_incremental_gb300 import _lib
    lib = _lib.load()
    h = sc.cache._h
    q = torch.zeros((2, 4, 8, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((2, 4, 2, 64), dtype=torch.bfloat16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    before = _snapshot(sc)

    def append(layer=0, Hq=8, C=4, n=(1, 1), rows=None, Bs=2, qp=None, out=None):
        return lib.kv_append(h, layer, qp if qp is not None else q.data_ptr(), k.data_ptr(),
                             k.data_ptr(), Hq, C, _i32(n), None if rows is None else _i32(rows),
                             Bs, out if out is not None else q.data_ptr(), stream)

    E = _lib
    assert append(layer=2) == E.KV_ERR_ARG                       # no such layer
    assert append(layer=-1) == E.KV_ERR_ARG
    assert append(Hq=4) == E.KV_ERR_ARG                          # Hq differs from the cache
    assert append(C=0) == E.KV_ERR_ARG
    assert append(n=(5, 1)) == E.KV_ERR_ARG                      # n_new > C
    assert append(n=(-1, 1)) == E.KV_ERR_ARG
    assert append(rows=(1, 1)) == E.KV_ERR_ARG                   # duplicate rows
    assert append(rows=(0, 4)) == E.KV_ERR_ARG                   # row out of range
    assert append(Bs=5, n=(1,) * 5) == E.KV_ERR_ARG              # more rows than the cache
    assert append(rows=(3, 0), n=(2, 1)) == E.KV_ERR_FULL        # row 3 holds 39 of 40
    assert append(qp=q.data_ptr() + 2) == E.KV_ERR_ARG           # misaligned pointer
    assert lib.kv_append(h, 0, None, None, None, 8, 4, _i32([1, 0]), None, 2, None,
                         stream) == E.KV_ERR_ARG                 # null tensors with work to do
    assert lib.kv_advance(h, _i32([1, 1]), _i32([3, 3]), 2, stream) == E.KV_ERR_ARG
    assert lib.kv_advance(h, _i32([2]), _i32([3]), 1, stream) == E.KV_ERR_FULL
    assert lib.kv_reset(h, _i32([0, 0]), 2, stream) == E.KV_ERR_ARG
    assert lib.kv_reset(h, _i32([7]), 1, stream) == E.KV_ERR_ARG
    assert lib.kv_debug_ptrs(h, 9, None, None, None) == E.KV_ERR_ARG
    after = _snapshot(sc)
    assert after[1] == before[1]
    assert all(np.array_equal(x, y) for x, y in zip(before[0], after[0]))
    # nothing to do is not an error, and leaves everything as it was
    assert append(n=(0, 0)) == E.KV_OK
    assert lib.kv_advance(h, _i32([0, 0]), None, 2, stream) == E.KV_OK
    assert lib.kv_reset(h, _i32([]), 0, stream) == E.KV_OK
    assert _snapshot(sc)[1] == before[1]
    # the cache still works after the rejections
    sc.step([1, 1, 1, 1], C=1, check_state=True)


def test_binding_guards_dtype_shape_and_device(sc):
    import torch
    import kv_cache_incremental_gb300 as kvi
    q = torch.zeros((2, 1, 8, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((2, 1, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TypeError):
        sc.cache.append(0, q.half(), k, k, [1, 1])
    with pytest.raises(ValueError):
        sc.cache.append(0, q, k[:, :, :1], k, [1, 1])
    with pytest.raises(ValueError):
        sc.cache.append(0, q.cpu(), k, k, [1, 1])
    with pytest.raises(ValueError):
        sc.cache.append(0, q, k, k, [1])
    q2 = torch.zeros((2, 2, 8, 64), dtype=torch.bfloat16, device="cuda")
    k2 = torch.zeros((2, 2, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvi.KVCacheFull):
        sc.cache.append(0, q2, k2, k2, [2, 1], rows=[3, 0])   # 39 + 2 > 40
    assert sc.cache.lens == [10, 3, 0, 39]


def test_create_rejects_bad_layouts_and_reports_memory():
    import kv_cache_incremental_gb300 as kvi
    for kw in (dict(Hq=6, Hk=4), dict(D=96), dict(Hq=64, Hk=2), dict(W=0, layer_kinds=[1])):
        args = dict(B=2, max_len=16, Hq=4, Hk=2, D=64, W=4, layer_kinds=[0])
        args.update(kw)
        with pytest.raises(kvi.KVError):
            kvi.KVCache(**args)
    c = kvi.KVCache(B=3, max_len=64, Hq=4, Hk=2, D=16 * 4, W=8, layer_kinds=[0, 1])
    # K+V bytes: global [3][2][65][64] + ring [3][2][9][64], bf16, times two (K and V)
    assert c.nbytes() == 2 * 3 * 2 * 65 * 64 * 2 + 2 * 3 * 2 * 9 * 64 * 2
    assert c.R == 8 and c.lens == [0, 0, 0]
    c.close()
