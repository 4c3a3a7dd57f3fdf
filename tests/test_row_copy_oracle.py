"""Prefix reuse and row export / import against the oracle.

After every kv_copy_rows (fork, prefix reuse, in-place truncation, grow-with-copy into a
cache of another max_len) and every kv_import_row, the destination row's history is the
source's first `keep` positions (the harness maps them back to the source's streams) and
then a fresh stream of its own.  The checks: the whole cache state -- K/V of every kept
position, ring slots, lpos, lens -- bit for bit against the oracle, and the outputs of
the decode steps and chunks that follow, element by element, against cache-free attention
over that history.  A ring copied into the wrong slots ("a silently rotated cache",
inkling ring-buffer PR, review of the change) keeps the right bytes but at the wrong
positions: check_state and every later window over it fail.
"""
import pytest

from harness import Scenario

pytestmark = pytest.mark.gpu


def test_fork_of_wrapped_rings_decodes_and_chunks_like_the_oracle():
    kw = dict(B=5, max_len=128, Hq=8, Hk=2, D=64, W=8, kinds=[1, 0, 1], seed=61)
    sc = Scenario(**kw)
    sc.step([37, 5, 0, 12, 64], C=64, check_state=True)     # rows 0, 4 wrapped 4-8 times
    sc.copy_rows(sc, src_rows=[0, 0], dst_rows=[2, 4])
    assert sc.cache.lens == [37, 5, 37, 12, 37]
    sc.check_state()
    for _ in range(4):
        sc.step([1] * 5, check_state=True)
    sc.step([7, 3, 20, 1, 9], C=20, check_state=True)       # chunks past W on copied rows


def test_prefix_reuse_and_truncation_like_the_oracle():
    kw = dict(B=4, max_len=96, Hq=8, Hk=2, D=64, W=32, kinds=[0, 1], seed=62)
    sc = Scenario(**kw)
    sc.step([30, 11, 0, 2], C=30, check_state=True)          # no ring wrapped (30 <= 32)
    sc.copy_rows(sc, src_rows=[0], dst_rows=[2], keep=[20])  # shared-prompt prefix
    sc.copy_rows(sc, src_rows=[0], dst_rows=[0], keep=[25])  # in-place truncation
    sc.copy_rows(sc, src_rows=[1], dst_rows=[3], keep=[0])   # an empty prefix
    assert sc.cache.lens == [25, 11, 20, 0]
    sc.check_state()
    sc.step([1, 1, 1, 1], check_state=True)
    sc.step([40, 2, 33, 17], C=40, check_state=True)         # rings wrap after the copy
    for _ in range(3):
        sc.step([1, 0, 1, 1], check_state=True)


def test_grow_with_copy_of_wrapped_rings_into_a_larger_cache():
    """The reviewer's case: rows whose rings wrapped move to a cache with another max_len
    (rings copied position by position, global rows linearly) and keep decoding."""
    kinds = [1, 0, 1, 0]
    small = Scenario(B=3, max_len=48, Hq=8, Hk=2, D=64, W=8, kinds=kinds, seed=63)
    small.step([40, 9, 3], C=40, check_state=True)
    big = Scenario(B=6, max_len=300, Hq=8, Hk=2, D=64, W=8, kinds=kinds, seed=64)
    big.step([5, 0, 0, 0, 0, 0], C=5)                        # row 0 is overwritten below
    big.copy_rows(small, src_rows=[0, 1, 2], dst_rows=[5, 0, 3])
    assert big.cache.lens == [9, 0, 0, 3, 0, 40]
    big.check_state()
    for _ in range(10):
        big.step([1, 0, 0, 1, 0, 1], check_state=True)
    big.step([30, 0, 0, 12, 0, 64], C=64, check_state=True)


def test_grow_with_copy_between_caches_with_different_ring_sizes():
    """A cache whose max_len is below W keeps R = max_len ring slots; its rows copied into a
    cache with R = W land at slot p % W and decode past the old ring size."""
    tiny = Scenario(B=2, max_len=6, Hq=8, Hk=2, D=64, W=8, kinds=[1, 0], seed=65)
    tiny.step([6, 4], C=6, check_state=True)
    assert tiny.cache.R == 6
    big = Scenario(B=3, max_len=100, Hq=8, Hk=2, D=64, W=8, kinds=[1, 0], seed=66)
    assert big.cache.R == 8
    big.copy_rows(tiny, src_rows=[0, 1], dst_rows=[1, 2])
    big.check_state()
    for _ in range(10):
        big.step([0, 1, 1], check_state=True)
    big.step([0, 9, 17], C=17, check_state=True)


def test_export_import_like_the_oracle():
    kinds = [0, 1, 1]
    a = Scenario(B=3, max_len=80, Hq=8, Hk=2, D=64, W=16, kinds=kinds, seed=67)
    a.step([50, 16, 7], C=50, check_state=True)
    b = Scenario(B=2, max_len=120, Hq=8, Hk=2, D=64, W=16, kinds=kinds, seed=68)
    b.import_row(1, a.cache.export_row(0), keep=50, src=a, src_row=0)     # wrapped rings
    b.import_row(0, a.cache.export_row(1, keep=10), keep=10, src=a, src_row=1)
    assert b.cache.lens == [10, 50]
    b.check_state()
    for _ in range(3):
        b.step([1, 1], check_state=True)
    b.step([12, 5], C=12, check_state=True)
    a.step([1, 1, 1], check_state=True)                       # the source is unchanged


def test_hybrid_copies_and_export_import_like_the_oracle():
    kinds = [2, 3, 1, 2]
    kw = dict(B=5, max_len=160, Hq=8, Hk=2, D=64, W=10, kinds=kinds, seed=69)
    sc = Scenario(**kw)
    sc.step([37, 8, 0, 64, 5], C=64, check_state=True)
    sc.copy_rows(sc, src_rows=[0, 0], dst_rows=[2, 4])       # whole rows (rings wrapped)
    sc.copy_rows(sc, src_rows=[1], dst_rows=[1], keep=[6])   # truncation of an unwrapped row
    sc.check_state()
    other = Scenario(**dict(kw, B=2, max_len=200, seed=70))
    other.import_row(1, sc.cache.export_row(3), keep=64, src=sc, src_row=3)
    other.check_state()
    for _ in range(3):
        sc.step([1, 1, 1, 1, 1], check_state=True)
        other.step([0, 1], check_state=True)
    sc.step([11, 2, 0, 5, 30], C=30, check_state=True)
    other.step([4, 20], C=20, check_state=True)


def test_paged_copies_and_import_like_the_oracle():
    kw = dict(B=4, max_len=200, Hq=8, Hk=2, D=64, W=16, kinds=[0, 1], seed=71)
    d = Scenario(**kw)
    p = Scenario(**dict(kw, seed=72), paged_blocks=60)
    d.step([40, 17, 3, 90], C=90, check=False)
    p.step([40, 17, 3, 90], C=90, check=False)
    p.copy_rows(d, src_rows=[3], dst_rows=[2])               # dense -> paged
    p.copy_rows(p, src_rows=[0], dst_rows=[1])               # paged -> paged, ring wrapped
    d.import_row(0, p.cache.export_row(2), keep=90, src=p, src_row=2)   # paged -> dense
    p.check_state()
    d.check_state()
    for _ in range(3):
        p.step([1, 1, 1, 1], check_state=True)
        d.step([1, 0, 0, 1], check_state=True)
    p.step([9, 33, 2, 20], C=33, check_state=True)           # crosses into new blocks


def test_paged_truncation_and_prefix_like_the_oracle():
    """Global layers only (no ring, so any prefix is present): truncation gives blocks back,
    a prefix shares the source's full blocks, and the rows then grow into fresh blocks."""
    p = Scenario(B=3, max_len=256, Hq=8, Hk=2, D=128, kinds=[0, 0], seed=73, paged_blocks=40)
    p.step([100, 37, 0], C=100, check=False)
    free = p.cache.free_blocks
    p.copy_rows(p, src_rows=[0], dst_rows=[0], keep=[33])    # 7 blocks -> 3
    assert p.cache.free_blocks == free + 4
    p.copy_rows(p, src_rows=[1], dst_rows=[2], keep=[17])
    p.check_state()
    for _ in range(3):
        p.step([1, 1, 1], check_state=True)
    p.step([64, 5, 48], C=64, check_state=True)
