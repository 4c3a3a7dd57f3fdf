"""Paged cache (kv_cache_create_paged): global layers in a pool of 16-position blocks.

The same scenarios as the dense parity tests run on paged caches against the oracle
(outputs within tolerance, cache contents, ring state and lens bit for bit), a paged
and a dense cache fed the same inputs agree bit for bit, pool exhaustion is refused
without any change, and forks inside a paged cache share the prefix's blocks.
"""
import numpy as np
import pytest

from harness import Scenario, torch_to_bits

pytestmark = pytest.mark.gpu


def test_paged_config1_tiny_and_chunking():
    sc = Scenario(B=2, max_len=128, Hq=4, Hk=2, D=64, seed=1, paged_blocks=16)
    sc.step([5, 9], C=9, check_state=True)
    sc.step([5, 0], C=5, check_state=True)
    sc.step([5, 0], C=5, check_state=True)
    sc.step([2, 0], C=2, check_state=True)
    for _ in range(8):
        sc.step([1, 1], C=1, check_state=True)
    assert sc.lens == [25, 17]
    assert len(sc.cache.block_table(0)) == 2 and len(sc.cache.block_table(1)) == 2


def test_paged_ring_mix_multi_chunk_and_splits():
    """Sliding rings stay dense while the global layer is paged: prefills of several
    sub-chunks, long decodes with several splits, GQA groups of 4."""
    sc = Scenario(B=3, max_len=1600, Hq=16, Hk=4, D=128, W=40, kinds=[1, 0, 1],
                  seed=4, paged_blocks=300)
    sc.step([70, 3, 130], C=130, check_state=True)
    for _ in range(3):
        sc.step([1, 1, 1], C=1)
    lens_target = [1500, 700, 200]
    while max(t - l for t, l in zip(lens_target, sc.lens)) > 0:
        n = [min(64, max(0, t - l)) for t, l in zip(lens_target, sc.lens)]
        sc.step(n, C=64, check=False)
    sc.check_state()
    for _ in range(3):
        sc.step([1, 1, 1], C=1)
    sc.step([1, 0, 20], C=20, check_state=True)


def test_paged_rows_subset_resets_reuse_blocks():
    """Resets return blocks; later appends of other rows take them again."""
    sc = Scenario(B=6, max_len=200, Hq=4, Hk=2, D=64, W=16, kinds=[1, 0], seed=6,
                  paged_blocks=20)
    sc.step([10, 20, 0, 5], rows=[4, 0, 2, 5], C=20, check_state=True)
    sc.step([1, 1], rows=[0, 5], C=1, check_state=True)
    free_before = sc.cache.free_blocks
    sc.step([3, 1, 30], rows=[5, 4, 1], C=30, resets=[4], check_state=True)
    sc.step([0, 0], rows=[1, 2], C=4, check_state=True)
    sc.step([17], rows=[3], C=17, resets=[3], check_state=True)
    sc.step([40], rows=[0], C=40, resets=[0], check_state=True)
    used = sum(len(sc.cache.block_table(b)) for b in range(6))
    assert used + sc.cache.free_blocks == 20
    assert free_before >= 0


def test_paged_equals_dense_bit_for_bit():
    import torch
    kw = dict(B=4, max_len=600, Hq=32, Hk=8, D=128, W=64, kinds=[0, 1, 0], seed=12)
    d, p = Scenario(**kw), Scenario(**kw, paged_blocks=4 * 38)
    for sc in (d, p):
        sc.step([64, 33, 1, 50], C=64, check=False)
        sc.step([64, 64, 64, 64], C=64, check=False)
        sc.step([9, 0, 64, 2], C=64, check=False)
    for _ in range(4):
        od = d.step([1, 1, 1, 1], C=1, check=False)
        op = p.step([1, 1, 1, 1], C=1, check=False)
        for (qa, a), (qb, b) in zip(od, op):
            assert np.array_equal(torch_to_bits(a), torch_to_bits(b))
    oc = d.step([30, 1, 0, 64], C=64, check=False)
    pc = p.step([30, 1, 0, 64], C=64, check=False)
    for (qa, a), (qb, b) in zip(oc, pc):
        assert np.array_equal(torch_to_bits(a), torch_to_bits(b))
    for layer in range(3):
        for x, y in zip(d.cache.storage(layer), p.cache.storage(layer)):
            xb, yb = torch_to_bits(x), torch_to_bits(y)
            for b in range(4):
                L = d.lens[b]
                n = min(L, d.cache.R) if kw["kinds"][layer] == 1 else L
                assert np.array_equal(xb[b, :, :n], yb[b, :, :n])
    p.check_state()


def test_pool_exhaustion_changes_nothing():
    import torch
    import kv_cache_incremental_gb300 as kvi
    sc = Scenario(B=3, max_len=128, Hq=4, Hk=2, D=64, kinds=[0, 0], seed=3, paged_blocks=5)
    sc.step([40, 30, 0], C=40, check_state=True)      # 3 + 2 blocks: the pool is used up
    assert sc.cache.free_blocks == 0
    before = [torch_to_bits(x) for x in sc.cache.storage(0)]
    q = torch.zeros((1, 1, 4, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 1, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvi.KVPoolExhausted):
        sc.cache.append(0, q, k, k, [1], rows=[2])        # row 2 needs a first block
    torch.cuda.synchronize()
    after = [torch_to_bits(x) for x in sc.cache.storage(0)]
    assert all(np.array_equal(x, y) for x, y in zip(before, after))
    assert sc.cache.lens == [40, 30, 0]
    sc.step([1, 1], rows=[0, 1], C=1, check_state=True)  # 41, 31 fit in their blocks
    sc.step([5], rows=[2], C=5, resets=[1], check_state=True)   # row 1's blocks reused


def test_paged_step_graph_and_copies():
    """The decode-step graph, row copies between paged and dense caches, export/import."""
    import torch
    kw = dict(B=4, max_len=200, Hq=8, Hk=2, D=64, W=16, kinds=[0, 1], seed=17)
    d, p = Scenario(**kw), Scenario(**kw, paged_blocks=60)
    for sc in (d, p):
        sc.step([40, 17, 3, 90], C=90, check=False)
    # dense -> paged and paged -> paged copies, then identical decodes
    p.cache.copy_rows(d.cache, src_rows=[3], dst_rows=[2])
    p.cache.copy_rows(p.cache, src_rows=[0], dst_rows=[1])   # whole row (its ring wrapped)
    buf = p.cache.export_row(3)
    d.cache.import_row(0, buf, keep=90)
    assert p.cache.lens == [40, 40, 90, 90] and d.cache.lens == [90, 17, 3, 90]
    ref = [torch_to_bits(x) for x in d.cache.storage(0)]
    got = [torch_to_bits(x) for x in p.cache.storage(0)]
    for x, y in zip(ref, got):
        assert np.array_equal(x[3, :, :90], y[2, :, :90])
        assert np.array_equal(x[0, :, :90], y[3, :, :90])
    mk = lambda H: [torch.zeros((2, 1, H, 64), dtype=torch.bfloat16, device="cuda")
                    for _ in range(2)]
    bufs_d = (mk(8), mk(2), mk(2), mk(8))
    bufs_p = (mk(8), mk(2), mk(2), mk(8))
    gd = d.cache.step_graph(*bufs_d, rows=[0, 3])
    gp = p.cache.step_graph(*bufs_p, rows=[3, 2])
    gen = torch.Generator().manual_seed(0)
    for _ in range(20):                               # crosses into new blocks
        for layer in range(2):
            for i, H in enumerate((8, 2, 2)):
                x = torch.randn((2, 1, H, 64), generator=gen).to(torch.bfloat16).cuda()
                bufs_d[i][layer].copy_(x)
                bufs_p[i][layer].copy_(x)
        gd.launch()
        gp.launch()
        torch.cuda.synchronize()
        for layer in range(2):
            assert np.array_equal(torch_to_bits(bufs_d[3][layer]),
                                  torch_to_bits(bufs_p[3][layer]))
    assert p.cache.lens[3] == 110 and len(p.cache.block_table(3)) == 7
    gd.close()
    gp.close()


def _pool_accounting(sc):
    """Every pool block is free or held by some row, never both; a block that several rows
    hold lies below each holder's length (no append can write it)."""
    tables = [sc.cache.block_table(r) for r in range(sc.B)]
    held = {}
    for r, t in enumerate(tables):
        assert len(t) == (sc.lens[r] + 15) // 16
        for i, blk in enumerate(t):
            held.setdefault(blk, []).append((r, i))
    assert len(held) + sc.cache.free_blocks == sc.cache.paged_blocks
    for blk, holders in held.items():
        if len(holders) > 1:
            assert all(16 * (i + 1) <= sc.lens[r] for r, i in holders), (blk, holders)
    return tables


def test_shared_prefix_blocks_like_the_oracle():
    """Prefix sharing with reference-counted blocks ("Lab 07 -- KV cache and sampling",
    Stretch: prompts with the same 32-token system prompt share its blocks).  Forks inside
    one paged cache hold the source's full blocks of the prefix -- equal block ids, the pool
    giving only a partly filled last block -- and every row then decodes and prefills its
    own continuation like the oracle.  A row cut in place inside a block other rows hold
    takes a copy of it first; resets and imports let go of shared blocks, which return to
    the pool with their last holder."""
    sc = Scenario(B=6, max_len=256, Hq=8, Hk=2, D=64, W=128, kinds=[0, 1, 0], seed=81,
                  paged_blocks=64)   # (rings that do not wrap: any prefix can be copied)
    sc.step([40, 0, 0, 0, 0, 0], C=40, check=False)        # row 0: a 40-token prompt
    t0 = sc.cache.block_table(0)
    free = sc.cache.free_blocks
    # rows 1 and 2: its 32-token system prompt (two full blocks); row 3: all 40 tokens
    sc.copy_rows(sc, src_rows=[0, 0, 0], dst_rows=[1, 2, 3], keep=[32, 32, 40])
    tables = _pool_accounting(sc)
    assert tables[1] == tables[2] == t0[:2]
    assert tables[3][:2] == t0[:2] and tables[3][2] != t0[2]
    assert sc.cache.free_blocks == free - 1               # 8 blocks of prompts, 4 in the pool
    sc.check_state()
    for _ in range(2):
        sc.step([1, 1, 1, 1, 0, 0], check_state=True)
    sc.step([5, 17, 3, 30, 0, 0], C=30, check_state=True)  # into blocks of their own
    tables = _pool_accounting(sc)
    assert all(tables[r][:2] == t0[:2] for r in (1, 2, 3))
    # row 0 cut to 20 tokens in place: its second block, held by rows 1-3 too, is copied
    sc.copy_rows(sc, src_rows=[0], dst_rows=[0], keep=[20])
    tables = _pool_accounting(sc)
    assert tables[0][0] == t0[0] and tables[0][1] != t0[1]
    assert all(tables[r][1] == t0[1] for r in (1, 2, 3))
    sc.check_state()
    sc.step([12, 1, 1, 1, 0, 0], C=12, check_state=True)
    # a fork of a fork, then resets and an import over shared rows
    sc.copy_rows(sc, src_rows=[3], dst_rows=[4], keep=[33])
    tables = _pool_accounting(sc)
    assert tables[4][:2] == t0[:2]
    free = sc.cache.free_blocks
    own = len(tables[1]) - 2 + len(tables[2]) - 2
    sc.step([0, 0, 0, 0, 0, 0], resets=[1, 2], check=False)
    assert sc.cache.free_blocks == free + own            # t0[:2] still held by rows 3, 4
    sc.import_row(3, sc.cache.export_row(4), keep=33, src=sc, src_row=4)
    tables = _pool_accounting(sc)
    assert not set(tables[3]) & set(tables[4])           # an import writes blocks of its own
    sc.check_state()
    sc.step([3, 2, 1, 1, 1, 4], C=4, check_state=True)
    sc.step([0, 0, 0, 0, 0, 0], resets=[0, 1, 2, 3, 4, 5], check=False)
    _pool_accounting(sc)
    assert sc.cache.free_blocks == 64


def test_shared_prefix_memory_saved():
    """The pool memory prefix sharing saves: eight requests with a common 32-token system
    prompt hold its two blocks once instead of eight times, and a fork of a 100-token row
    takes one block (its partly filled last one) instead of seven."""
    sc = Scenario(B=9, max_len=256, Hq=8, Hk=2, D=64, kinds=[0, 0], seed=82, paged_blocks=64)
    sc.step([32] + [0] * 8, C=32, check=False)             # the system prompt, in row 0
    free = sc.cache.free_blocks
    sc.copy_rows(sc, src_rows=[0] * 8, dst_rows=list(range(1, 9)))
    assert sc.cache.free_blocks == free                   # 8 x 2 blocks held, none taken
    sc.step([0] + [20] * 8, C=20, check_state=True)        # each request's own continuation
    used = 64 - sc.cache.free_blocks
    copied = sum((sc.lens[r] + 15) // 16 for r in range(9))
    assert (used, copied) == (2 + 8 * 2, 2 + 8 * 4)       # 18 blocks held instead of 34
    block_bytes = 2 * 2 * sc.Hk * 16 * sc.D * 2            # 2 layers x (K, V) x [Hk][16][D] bf16
    assert (copied - used) * block_bytes == 16 * 16384
    sc.copy_rows(sc, src_rows=[1], dst_rows=[0], keep=[52])  # 52 = 3 full blocks + 4
    assert 64 - sc.cache.free_blocks == used + 1           # row 0's old blocks: still held
