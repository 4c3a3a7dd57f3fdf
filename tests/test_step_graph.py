"""Decode-step graph (kv_step_graph_*) against the kv_append / kv_advance path.

The graph replays the same kernels with the parameters kv_append would pass, so its
outputs, cache contents, ring slots, lpos and lens must equal the direct path's bit for
bit; the direct path is itself checked against the oracle.
"""
import numpy as np
import pytest

from harness import Scenario, bf16_bits_to_torch, torch_to_bits

pytestmark = pytest.mark.gpu


def _buffers(sc, Bs):
    import torch
    mk = lambda H: [torch.zeros((Bs, 1, H, sc.D), dtype=torch.bfloat16, device=sc.dev)
                    for _ in sc.kinds]
    return mk(sc.Hq), mk(sc.Hk), mk(sc.Hk), mk(sc.Hq)


def _graph_step(sc, g, bufs, rows):
    """One replay: this step's inputs into the graph's buffers, launch, host bookkeeping."""
    import torch
    qb, kb, vb, ob = bufs
    ones = [1] * len(rows)
    qs = []
    for layer in range(len(sc.kinds)):
        q, k, v = sc.chunk_inputs(layer, rows, ones, 1)
        qb[layer].copy_(bf16_bits_to_torch(q, sc.dev))
        kb[layer].copy_(bf16_bits_to_torch(k, sc.dev))
        vb[layer].copy_(bf16_bits_to_torch(v, sc.dev))
        qs.append(q)
    g.launch()
    torch.cuda.synchronize()
    outs = [torch_to_bits(o) for o in ob]
    for b in rows:
        sc.lens[b] += 1
    return qs, outs


def _same_state(a, b):
    """Live region of every layer, lpos and lens equal between the two caches."""
    assert a.cache.lens == b.cache.lens
    for layer in range(len(a.kinds)):
        sa = [torch_to_bits(t) for t in a.cache.storage(layer)]
        sb = [torch_to_bits(t) for t in b.cache.storage(layer)]
        for r in range(a.B):
            L = a.lens[r]
            n = min(L, a.cache.R) if a.kinds[layer] == 1 else L
            for xa, xb in zip(sa, sb):
                assert np.array_equal(xa[r, :, :n], xb[r, :, :n]), (layer, r)
    if a.cache.lpos() is not None:
        assert np.array_equal(a.cache.lpos().cpu().numpy(), b.cache.lpos().cpu().numpy())


@pytest.mark.parametrize("Hq,Hk,D", [(8, 2, 64), (32, 2, 128)])
def test_graph_equals_append_advance(Hq, Hk, D):
    """Sliding and global layers, rows at different lengths (one empty, one wrapping the
    ring), six replays: bit-identical to per-layer kv_append + kv_advance."""
    kw = dict(B=5, max_len=192, Hq=Hq, Hk=Hk, D=D, W=16, kinds=[1, 0, 1], seed=21)
    a, b = Scenario(**kw), Scenario(**kw)
    fill = [20, 33, 7, 0, 64]
    a.step(fill, C=64, check=False)
    b.step(fill, C=64, check=False)
    rows = list(range(5))
    bufs = _buffers(b, len(rows))
    g = b.cache.step_graph(*bufs, rows=rows)
    for _ in range(6):
        outs_a = a.step([1] * 5, rows, C=1)            # checked against the oracle
        qs, outs_b = _graph_step(b, g, bufs, rows)
        for layer in range(3):
            assert np.array_equal(torch_to_bits(outs_a[layer][1]), outs_b[layer]), layer
    _same_state(a, b)
    b.check_state()
    g.close()


def test_graph_row_subset_and_reset_between_launches():
    """A subset of rows in a non-trivial order; other rows are untouched; a reset of a
    graph row between launches is planned from its new length."""
    kw = dict(B=6, max_len=160, Hq=8, Hk=2, D=64, W=8, kinds=[0, 1], seed=5)
    a, b = Scenario(**kw), Scenario(**kw)
    fill = [9, 40, 3, 17, 25, 1]
    a.step(fill, C=40, check=False)
    b.step(fill, C=40, check=False)
    rows = [4, 1, 3]
    bufs = _buffers(b, len(rows))
    g = b.cache.step_graph(*bufs, rows=rows)
    for it in range(4):
        if it == 2:
            for sc in (a, b):
                sc.cache.reset([1])
                sc.mark_reset([1])
        outs_a = a.step([1] * 3, rows, C=1)
        qs, outs_b = _graph_step(b, g, bufs, rows)
        for layer in range(2):
            assert np.array_equal(torch_to_bits(outs_a[layer][1]), outs_b[layer])
    assert b.cache.lens[0] == 9 and b.cache.lens[2] == 3 and b.cache.lens[5] == 1
    _same_state(a, b)
    b.check_state()
    g.close()


def test_graph_set_buffers_alternating():
    """Two buffer sets, swapped before every launch: still the direct path's results."""
    kw = dict(B=4, max_len=128, Hq=16, Hk=4, D=64, W=12, kinds=[0, 1, 1], seed=13)
    a, b = Scenario(**kw), Scenario(**kw)
    fill = [30, 5, 12, 19]
    a.step(fill, C=30, check=False)
    b.step(fill, C=30, check=False)
    rows = [0, 1, 2, 3]
    sets = [_buffers(b, 4), _buffers(b, 4)]
    g = b.cache.step_graph(*sets[1], rows=rows)
    for it in range(5):
        g.set_buffers(*sets[it % 2])
        outs_a = a.step([1] * 4, rows, C=1)
        qs, outs_b = _graph_step(b, g, sets[it % 2], rows)
        for layer in range(3):
            assert np.array_equal(torch_to_bits(outs_a[layer][1]), outs_b[layer])
    _same_state(a, b)
    g.close()


def test_graph_full_row_raises_without_state_change():
    import kv_cache_incremental_gb300 as kvi
    sc = Scenario(B=2, max_len=24, Hq=4, Hk=2, D=64, W=8, kinds=[1, 0], seed=9)
    sc.step([23, 10], C=23, check=False)
    bufs = _buffers(sc, 2)
    g = sc.cache.step_graph(*bufs)
    _graph_step(sc, g, bufs, [0, 1])                    # row 0 reaches max_len
    before = sc.cache.lens
    with pytest.raises(kvi.KVCacheFull):
        g.launch()
    assert sc.cache.lens == before == [24, 11]
    sc.check_state()
    g.close()


def test_graph_argument_errors():
    import torch
    import kv_cache_incremental_gb300 as kvi
    sc = Scenario(B=3, max_len=32, Hq=4, Hk=2, D=64, kinds=[0], seed=1)
    q, k, v, o = _buffers(sc, 2)
    with pytest.raises(kvi.KVError):
        sc.cache.step_graph(q, k, v, o, rows=[1, 1])    # duplicate rows
    with pytest.raises(kvi.KVError):
        sc.cache.step_graph(q, k, v, o, rows=[0, 3])    # row out of range
    with pytest.raises(ValueError):
        sc.cache.step_graph(q, k, v, o + o)             # one buffer set per layer
    bad = [torch.zeros((2, 2, 4, 64), dtype=torch.bfloat16, device=sc.dev)]
    with pytest.raises(ValueError):
        sc.cache.step_graph(bad, k, v, o)               # not one token per row
    g = sc.cache.step_graph(q, k, v, o, rows=[2, 0])
    sc.cache.close()                                    # closes the graph first
    assert g._h is None
