"""Hybrid layers (kv_append_hybrid): one softmax over a layer group's global keys at every
position <= p and the layer's own local keys in the window p-W+1..p.

The group's full layer (kind 2) writes the group's global K/V; the local layers (kind 3)
read it; every hybrid layer keeps its own ring.  Outputs are checked against the oracle's
hybrid attention within tolerance; the group cache, the rings, lpos and lens bit for bit.
Decode rows (split-K over both segments, the new global key appended only by the full
layer), chunked prefill (three key segments: group cache, ring, chunk) and the ring commit
are all on the path.
"""
import numpy as np
import pytest

from harness import Scenario, torch_to_bits

pytestmark = pytest.mark.gpu


def test_hybrid_tiny_prefill_then_decode():
    sc = Scenario(B=3, max_len=160, Hq=4, Hk=2, D=64, W=16, kinds=[2, 3, 3], seed=1)
    sc.step([5, 9, 2], C=9, check_state=True)
    sc.step([1, 1, 1], C=1, check_state=True)
    sc.step([20, 0, 1], C=20, check_state=True)    # crosses W; a decode row beside a chunk
    for _ in range(6):
        sc.step([1, 1, 1], C=1)
    sc.check_state()
    assert sc.lens == [32, 16, 10]


def test_hybrid_mixed_with_global_and_sliding_layers():
    """A layout with a global layer, a sliding layer and two hybrid groups (one full layer
    alone, one with two local layers); rows reset and restart."""
    sc = Scenario(B=4, max_len=300, Hq=8, Hk=2, D=64, W=24,
                  kinds=[0, 2, 3, 1, 2, 3, 3], seed=2)
    sc.step([70, 3, 0, 130], C=130, check_state=True)   # several 64-token sub-chunks
    for _ in range(3):
        sc.step([1, 1, 1, 1], C=1)
    sc.step([2, 40, 1, 0], C=40, resets=[2], check_state=True)
    sc.step([1, 1], rows=[3, 0], C=1, check_state=True)
    assert sc.max_ratio <= 1.0


@pytest.mark.parametrize("Hq,Hk", [(16, 4), (64, 8), (32, 2), (8, 8)])
def test_hybrid_d128_long_rows_split_decode(Hq, Hk):
    """D=128, long rows: the decode splits the group cache over several CTAs and adds the
    ring as its own split; tensor-core prefill over 128-key blocks of all three segments."""
    sc = Scenario(B=2, max_len=1400, Hq=Hq, Hk=Hk, D=128, W=40, kinds=[2, 3], seed=3)
    sc.step([200, 57], C=200, check_state=True)
    target = [1300, 640]
    while max(t - l for t, l in zip(target, sc.lens)) > 0:
        n = [min(64, max(0, t - l)) for t, l in zip(target, sc.lens)]
        sc.step(n, C=64, check=False)
    sc.check_state()
    for _ in range(3):
        sc.step([1, 1], C=1)
    sc.step([33, 1], C=33, check_state=True)


def test_hybrid_window_covers_whole_row():
    """W >= max_len: the ring never wraps and every local key stays visible."""
    sc = Scenario(B=2, max_len=48, Hq=4, Hk=1, D=64, W=64, kinds=[2, 3], seed=4)
    assert sc.cache.R == 48
    sc.step([30, 7], C=30, check_state=True)
    for _ in range(5):
        sc.step([1, 1], C=1)
    sc.step([13, 0], C=13, check_state=True)
    assert sc.lens[0] == 48


def test_hybrid_paged_equals_dense_bit_for_bit():
    import torch
    kw = dict(B=3, max_len=400, Hq=16, Hk=4, D=128, W=32, kinds=[2, 3, 0, 3], seed=5)
    d, p = Scenario(**kw), Scenario(**kw, paged_blocks=3 * 25)
    # kinds [2, 3, 0, 3]: the last local layer belongs to the group opened by layer 0
    for sc in (d, p):
        sc.step([64, 33, 1], C=64, check=False)
        sc.step([100, 64, 64], C=100, check=False)
    p.check_state()
    for _ in range(3):
        od = d.step([1, 1, 1], C=1)
        op = p.step([1, 1, 1], C=1, check=False)
        for (qa, a), (qb, b) in zip(od, op):
            assert np.array_equal(torch_to_bits(a), torch_to_bits(b))
    oc = d.step([30, 1, 9], C=30, check=False)
    pc = p.step([30, 1, 9], C=30, check=False)
    for (qa, a), (qb, b) in zip(oc, pc):
        assert np.array_equal(torch_to_bits(a), torch_to_bits(b))
    p.check_state()


def test_hybrid_refusals():
    import torch
    import kv_cache_incremental_gb300 as kvi
    with pytest.raises(kvi.KVError):
        kvi.KVCache(2, 32, 4, 2, 64, 8, [3, 2])        # a local layer before any full layer
    sc = Scenario(B=2, max_len=64, Hq=4, Hk=2, D=64, W=8, kinds=[2, 3, 0], seed=6)
    sc.step([10, 3], C=10, check=False)
    z = lambda H, C=1: torch.zeros((2, C, H, 64), dtype=torch.bfloat16, device="cuda")
    q, k = z(4), z(2)
    c = sc.cache
    with pytest.raises(kvi.KVError):
        c.append(0, q, k, k, [1, 1])                    # hybrid layer through kv_append
    with pytest.raises(kvi.KVError):
        c.append_hybrid(2, q, k, k, [1, 1])             # a global layer
    with pytest.raises(kvi.KVError):
        c.append_hybrid(0, q, k, k, [1, 1])             # full layer without global keys
    with pytest.raises(kvi.KVError):
        c.append_hybrid(1, q, k, k, [1, 1])             # local layer before its full layer
    c.append_hybrid(0, q, k, k, [1, 0], k_global=k, v_global=k)
    with pytest.raises(kvi.KVError):
        c.append_hybrid(1, q, k, k, [1, 0], k_global=k, v_global=k)  # global keys on local
    with pytest.raises(kvi.KVError):
        c.append_hybrid(1, q, k, k, [1, 1])             # other tokens than the full layer's
    c.append_hybrid(1, q, k, k, [1, 0])
    torch.cuda.synchronize()
    with pytest.raises(ValueError):                     # global buffers of the full layer
        c.step_graph([q] * 3, [k] * 3, [k] * 3, [q] * 3)
    assert c.lens == [10, 3]


def _bufs(sc, Bs):
    import torch
    mk = lambda H: torch.zeros((Bs, 1, H, sc.D), dtype=torch.bfloat16, device=sc.dev)
    q = [mk(sc.Hq) for _ in sc.kinds]
    k = [mk(sc.Hk) for _ in sc.kinds]
    v = [mk(sc.Hk) for _ in sc.kinds]
    o = [mk(sc.Hq) for _ in sc.kinds]
    kg = [mk(sc.Hk) if kind == 2 else None for kind in sc.kinds]
    vg = [mk(sc.Hk) if kind == 2 else None for kind in sc.kinds]
    return q, k, v, o, kg, vg


def _state(c, kinds, row):
    """(positions, K bits, V bits) of every storage unit of a row: a layer's own storage,
    then its hybrid ring."""
    L, out = c.lens[row], []
    for layer, kind in enumerate(kinds):
        views = []
        if kind in (0, 2):
            views.append((c.storage(layer), False))
        if kind == 1:
            views.append((c.storage(layer), True))
        if kind in (2, 3):
            views.append((c.ring_storage(layer), True))
        for (K, V), ring in views:
            Kb, Vb = torch_to_bits(K)[row], torch_to_bits(V)[row]
            pos = np.arange(max(0, L - c.R) if ring else 0, L)
            slots = pos % c.R if ring else pos
            out.append((pos, Kb[:, slots], Vb[:, slots]))
    return out


def _same(a, ra, b, rb, kinds):
    assert a.lens[ra] == b.lens[rb]
    for x, y in zip(_state(a, kinds, ra), _state(b, kinds, rb)):
        for u, w in zip(x, y):
            assert np.array_equal(u, w)


def test_hybrid_step_graph_equals_append():
    """Graph replays on a layout with global, sliding and hybrid layers: outputs, group
    caches, rings, lpos and lens bit for bit equal to kv_append(_hybrid) + kv_advance."""
    import torch
    from harness import bf16_bits_to_torch
    kw = dict(B=4, max_len=200, Hq=16, Hk=4, D=64, W=12, kinds=[2, 3, 0, 1, 2, 3], seed=41)
    a, b = Scenario(**kw), Scenario(**kw)
    for sc in (a, b):
        sc.step([30, 3, 17, 0], C=30, check=False)
    rows = [3, 0, 2]
    q, k, v, o, kg, vg = _bufs(b, len(rows))
    g = b.cache.step_graph(q, k, v, o, rows=rows, k_global=kg, v_global=vg)
    ones = [1] * len(rows)
    for _ in range(5):
        outs_a = a.step(ones, rows, C=1)                 # checked against the oracle
        for layer, kind in enumerate(b.kinds):
            qq, kk, vv = b.chunk_inputs(layer, rows, ones, 1)
            for dst, src in ((q, qq), (k, kk), (v, vv)):
                dst[layer].copy_(bf16_bits_to_torch(src, b.dev))
            if kind == 2:
                gk, gvv = b.global_inputs(layer, rows, ones, 1)
                kg[layer].copy_(bf16_bits_to_torch(gk, b.dev))
                vg[layer].copy_(bf16_bits_to_torch(gvv, b.dev))
        g.launch()
        torch.cuda.synchronize()
        for r in rows:
            b.lens[r] += 1
        for layer in range(len(b.kinds)):
            assert np.array_equal(torch_to_bits(outs_a[layer][1]), torch_to_bits(o[layer]))
    for r in range(4):
        _same(a.cache, r, b.cache, r, b.kinds)
    assert np.array_equal(a.cache.lpos().cpu().numpy(), b.cache.lpos().cpu().numpy())
    b.check_state()
    # a local layer may follow its full layer again after the graph's steps
    b.step([2, 1], rows=[0, 1], C=2, check_state=True)
    g.close()


def test_hybrid_copies_and_export_import():
    """Fork rows whose rings have wrapped, truncate an unwrapped row, move a row to another
    cache through export / import: states equal position by position, and rows sharing a
    state decode identically."""
    import torch
    kinds = [2, 3, 1, 2]
    kw = dict(B=5, max_len=160, Hq=8, Hk=2, D=64, W=10, kinds=kinds, seed=43)
    sc = Scenario(**kw)
    sc.step([37, 8, 0, 64, 5], C=64, check_state=True)
    c = sc.cache
    c.copy_rows(c, src_rows=[0, 0], dst_rows=[2, 4])      # whole rows (rings wrapped)
    c.copy_rows(c, src_rows=[1], dst_rows=[1], keep=[6])   # truncation of an unwrapped row
    assert c.lens == [37, 6, 37, 64, 37]
    for d in (2, 4):
        _same(c, 0, c, d, kinds)
    other = Scenario(**dict(kw, B=2, max_len=200)).cache
    buf = c.export_row(3)
    other.import_row(1, buf, keep=64)
    _same(c, 3, other, 1, kinds)
    # identical inputs -> identical outputs for rows 0, 2, 4
    gen = torch.Generator().manual_seed(0)
    for _ in range(3):
        outs = []
        for layer, kind in enumerate(kinds):
            mk = lambda H: torch.randn((1, 1, H, 64), generator=gen).to(torch.bfloat16).expand(
                3, -1, -1, -1).contiguous().cuda()
            q, kl, vl = mk(8), mk(2), mk(2)
            kg, vg = (mk(2), mk(2)) if kind == 2 else (None, None)
            if kind in (2, 3):
                o = c.append_hybrid(layer, q, kl, vl, [1, 1, 1], k_global=kg, v_global=vg,
                                    rows=[0, 2, 4])
            else:
                o = c.append(layer, q, kl, vl, [1, 1, 1], rows=[0, 2, 4])
            outs.append(torch_to_bits(o))
        c.advance([1, 1, 1], rows=[0, 2, 4])
        torch.cuda.synchronize()
        for x in outs:
            assert np.array_equal(x[0], x[1]) and np.array_equal(x[0], x[2])
    for d in (2, 4):
        _same(c, 0, c, d, kinds)


def test_hybrid_host_buffers_equal_device():
    """kv_append_hybrid_host (pinned and pageable buffers) gives the device path's bits."""
    import torch
    kinds = [2, 3]
    kw = dict(B=3, max_len=120, Hq=8, Hk=2, D=64, W=16, kinds=kinds, seed=44)
    a, b = Scenario(**kw), Scenario(**kw)
    for sc in (a, b):
        sc.step([20, 5, 40], C=40, check=False)
    gen = torch.Generator().manual_seed(1)
    for it, (n, C) in enumerate((([1, 1, 1], 1), ([9, 0, 30], 30), ([1, 2, 1], 2))):
        pin = it % 2 == 0
        for layer, kind in enumerate(kinds):
            mk = lambda H: torch.randn((3, C, H, 64), generator=gen).to(torch.bfloat16)
            q, kl, vl = mk(8), mk(2), mk(2)
            kg, vg = (mk(2), mk(2)) if kind == 2 else (None, None)
            dev = lambda x: None if x is None else x.cuda()
            od = a.cache.append_hybrid(layer, dev(q), dev(kl), dev(vl), n, k_global=dev(kg),
                                       v_global=dev(vg))
            hp = (lambda x: None if x is None else x.pin_memory()) if pin else (lambda x: x)
            oh = torch.empty_like(q).pin_memory() if pin else torch.empty_like(q)
            b.cache.append_hybrid_host(layer, hp(q), hp(kl), hp(vl), n, k_global=hp(kg),
                                       v_global=hp(vg), out=oh)
            torch.cuda.synchronize()
            for i, m in enumerate(n):
                assert np.array_equal(torch_to_bits(od)[i, :m], torch_to_bits(oh)[i, :m])
        for sc in (a, b):
            sc.cache.advance(n)
    torch.cuda.synchronize()
    for r in range(3):
        _same(a.cache, r, b.cache, r, kinds)
