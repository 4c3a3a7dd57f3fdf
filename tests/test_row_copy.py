"""Prefix reuse and row export / import (kv_copy_rows, kv_export_row, kv_import_row).

A row's state is its length and, per layer, the K/V of the positions it keeps (all of
[0, lens) on a global layer, the last R on a sliding layer).  Checks: the copied state
equals the source's position by position, bit for bit; rows that share a state give
bit-identical outputs when fed identical inputs; refusals change nothing.
"""
import numpy as np
import pytest

from harness import torch_to_bits

pytestmark = pytest.mark.gpu


def _cache(B, max_len, W, kinds, Hq=8, Hk=2, D=64):
    import kv_cache_incremental_gb300 as kvi
    return kvi.KVCache(B, max_len, Hq, Hk, D, W, kinds, 1e4, 0)


def _rand(shape, gen):
    import torch
    return torch.randn(shape, generator=gen).to(torch.bfloat16).cuda()


def _feed(c, rows, n, gen, C=None, same=False):
    """Append n[i] tokens to rows[i] on every layer (identical inputs for all rows when
    same=True), then advance; returns the per-layer outputs as bits."""
    import torch
    Bs, C = len(rows), C or max(n)
    outs = []
    for layer in range(len(c.layer_kinds)):
        if same:
            q, k, v = (_rand((1, C, H, c.D), gen).expand(Bs, -1, -1, -1).contiguous()
                       for H in (c.Hq, c.Hk, c.Hk))
        else:
            q, k, v = (_rand((Bs, C, H, c.D), gen) for H in (c.Hq, c.Hk, c.Hk))
        outs.append(torch_to_bits(c.append(layer, q, k, v, list(n), rows=list(rows))))
    c.advance(list(n), rows=list(rows))
    torch.cuda.synchronize()
    return outs


def _state(c, row):
    """{layer: (positions, K bits [Hk][n][D], V bits)} of the positions the row keeps."""
    L, st = c.lens[row], {}
    for layer, kind in enumerate(c.layer_kinds):
        K, V = (torch_to_bits(t)[row] for t in c.storage(layer))
        pos = np.arange(max(0, L - c.R) if kind == 1 else 0, L)
        slots = pos % c.R if kind == 1 else pos
        st[layer] = (pos, K[:, slots], V[:, slots])
    return st


def _same_state(a, ra, b, rb):
    assert a.lens[ra] == b.lens[rb]
    sa, sb = _state(a, ra), _state(b, rb)
    for layer in sa:
        for x, y in zip(sa[layer], sb[layer]):
            assert np.array_equal(x, y), layer
    if a.lpos() is not None:
        la = a.lpos().cpu().numpy()[ra]
        lb = b.lpos().cpu().numpy()[rb]
        # the ring's (slot -> position) map is a function of the length alone
        if a.R == b.R:
            assert np.array_equal(la, lb)


def test_fork_then_identical_decodes():
    """Fork a row that has wrapped its rings into two others; the three then produce the
    same outputs for the same inputs, step after step."""
    import torch
    gen = torch.Generator().manual_seed(1)
    c = _cache(B=5, max_len=128, W=8, kinds=[1, 0, 1])
    _feed(c, [0, 1, 2, 3, 4], [37, 5, 0, 12, 64], gen, C=64)
    c.copy_rows(c, src_rows=[0, 0], dst_rows=[2, 4])
    assert c.lens == [37, 5, 37, 12, 37]
    for d in (2, 4):
        _same_state(c, 0, c, d)
    for _ in range(4):
        outs = _feed(c, [0, 2, 4], [1, 1, 1], gen, same=True)
        for o in outs:
            assert np.array_equal(o[0], o[1]) and np.array_equal(o[0], o[2])
    for d in (2, 4):
        _same_state(c, 0, c, d)
    assert c.lens[1] == 5 and c.lens[3] == 12   # rows not copied are untouched


def test_prefix_reuse_equals_shorter_fill():
    """A prefix copy (keep < lens) of a row equals a row filled with only that prefix; on a
    sliding cache this needs the source not to have wrapped (lens <= R)."""
    import torch
    gen = torch.Generator().manual_seed(2)
    c = _cache(B=4, max_len=96, W=32, kinds=[0, 1])
    # rows 0 and 1 get identical tokens: 30 for row 0, the first 20 of them for row 1
    import kv_cache_incremental_gb300 as kvi
    for layer in range(2):
        q, k, v = (_rand((1, 30, H, c.D), gen).expand(2, -1, -1, -1).contiguous()
                   for H in (c.Hq, c.Hk, c.Hk))
        c.append(layer, q, k, v, [30, 20], rows=[0, 1])
    c.advance([30, 20], rows=[0, 1])
    c.copy_rows(c, src_rows=[0], dst_rows=[2], keep=[20])
    _same_state(c, 1, c, 2)
    c.copy_rows(c, src_rows=[0], dst_rows=[0], keep=[25])   # in-place truncation
    assert c.lens[0] == 25
    outs = _feed(c, [1, 2], [1, 1], gen, same=True)
    for o in outs:
        assert np.array_equal(o[0], o[1])


def test_grow_with_copy_into_a_larger_cache():
    """Rows move into a cache with a larger max_len and another B (the rings copied by
    position, global prefixes linearly), then keep decoding like the originals."""
    import torch
    gen = torch.Generator().manual_seed(3)
    small = _cache(B=3, max_len=48, W=8, kinds=[1, 0, 1, 0])
    _feed(small, [0, 1, 2], [40, 9, 3], gen, C=40)
    big = _cache(B=6, max_len=300, W=8, kinds=[1, 0, 1, 0])
    big.copy_rows(small, src_rows=[0, 1, 2], dst_rows=[5, 0, 3])
    for s, d in ((0, 5), (1, 0), (2, 3)):
        _same_state(small, s, big, d)
    for _ in range(5):
        g_state = gen.get_state()
        o_small = _feed(small, [0, 1, 2], [1, 1, 1], gen)
        gen.set_state(g_state)
        o_big = _feed(big, [5, 0, 3], [1, 1, 1], gen)
        for a, b in zip(o_small, o_big):
            assert np.array_equal(a, b)


def test_export_import_round_trip():
    import torch
    gen = torch.Generator().manual_seed(4)
    a = _cache(B=3, max_len=80, W=16, kinds=[0, 1, 1])
    _feed(a, [0, 1, 2], [50, 16, 7], gen, C=50)
    b = _cache(B=2, max_len=80, W=16, kinds=[0, 1, 1])
    buf = a.export_row(0)
    b.import_row(1, buf, keep=50)
    _same_state(a, 0, b, 1)
    buf2 = a.export_row(1, keep=10)            # a prefix of a row that has not wrapped
    b.import_row(0, buf2, keep=10)
    a.copy_rows(a, [1], [2], keep=[10])
    _same_state(a, 2, b, 0)
    g_state = gen.get_state()
    oa = _feed(a, [0, 2], [1, 1], gen)
    gen.set_state(g_state)
    ob = _feed(b, [1, 0], [1, 1], gen)
    for x, y in zip(oa, ob):
        assert np.array_equal(x, y)


def test_refusals_change_nothing():
    import torch
    import kv_cache_incremental_gb300 as kvi
    gen = torch.Generator().manual_seed(5)
    c = _cache(B=4, max_len=64, W=8, kinds=[1, 0])
    _feed(c, [0, 1, 2, 3], [20, 6, 3, 1], gen, C=20)
    before = c.lens
    snap = [_state(c, r) for r in range(4)]
    other = _cache(B=2, max_len=64, W=16, kinds=[1, 0])
    for args in (
        dict(src=c, src_rows=[0], dst_rows=[1], keep=[15]),     # ring wrapped: not a prefix
        dict(src=c, src_rows=[1], dst_rows=[2], keep=[7]),      # keep > source length
        dict(src=c, src_rows=[0, 1], dst_rows=[2, 2]),          # duplicate destination
        dict(src=c, src_rows=[0, 2], dst_rows=[2, 3]),          # destination read by another pair
        dict(src=c, src_rows=[4], dst_rows=[0]),                # row out of range
    ):
        with pytest.raises(kvi.KVError):
            c.copy_rows(**args)
    with pytest.raises(kvi.KVError):
        other.copy_rows(c, [0], [0])                            # another layout (W)
    with pytest.raises(kvi.KVError):
        c.export_row(0, keep=15)                                # wrapped ring
    buf = c.export_row(1)
    with pytest.raises(kvi.KVError):
        c.import_row(2, buf, keep=5)                            # size does not match keep
    assert c.lens == before
    for r in range(4):
        now = _state(c, r)
        for layer in now:
            for x, y in zip(snap[r][layer], now[layer]):
                assert np.array_equal(x, y)
