"""The host planners of kv_append, run without a GPU through kv_plan_decode and
kv_plan_prefill: the split-K schedule of a decode launch and the key splits of chunked
prefill.  Every schedule must cover each row's keys exactly once in non-empty pieces,
give every split its own partial slots, respect the split caps, and spread a launch's
keys so that no CTA holds much more than its share; the kernel choice for chunk rows
follows the documented rule.
"""
import numpy as np
import pytest

import kv_cache_incremental_gb300 as kvi
from kv_cache_incremental_gb300 import KVError

GLOBAL, SLIDING, FULL, LOCAL = (kvi.KV_GLOBAL, kvi.KV_SLIDING, kvi.KV_HYBRID_FULL,
                                kvi.KV_HYBRID_LOCAL)
TILE = 64              # keys per tile
MAX_SPLITS = 32        # decode: splits per row over both segments
MAX_RING_SPLITS = 8    # decode: splits of a hybrid layer's ring
MIN_DECODE_TILES = 8   # decode: at most one split per this many tiles
MAX_PREFILL_SPLITS = 16
MIN_PREFILL_BLOCKS = 4  # prefill: at most one split per this many 128-key blocks
PART_VECS_PER_SM = 1024  # prefill: key-split partial vectors a cache reserves per SM
INF = 2**31 - 1


def tiles(keys):
    return -(-keys // TILE)


def decode_segments(kind, R, pos):
    """Keys of a decode row's segments: the layer storage, then a hybrid layer's ring."""
    ring = min(pos + 1, R)
    if kind == SLIDING:
        return ring, 0
    return pos + 1, ring if kind in (FULL, LOCAL) else 0


def check_decode(num_sms, Hq, Hk, D, R, kind, pos):
    p = kvi.plan_decode(num_sms, Hq, Hk, D, R, kind, pos)
    seg_tiles = [[tiles(k) for k in decode_segments(kind, R, x)] for x in pos]
    total_tiles = sum(sum(t) for t in seg_tiles)
    share = max(MIN_DECODE_TILES, -(-total_tiles * Hk // (num_sms * 2 * 4)))
    part = 0
    for i, (t0, t1) in enumerate(seg_tiles):
        ns, st, ns2, st2 = (p["n_splits"][i], p["split_tiles"][i], p["n_splits2"][i],
                            p["split_tiles2"][i])
        # segment caps: the ring's, then what the ring leaves to the storage segment
        for t, n, s, cap in ((t0, ns, st, MAX_SPLITS - ns2), (t1, ns2, st2, MAX_RING_SPLITS)):
            if t == 0:
                assert n == 0
                continue
            # n splits of s tiles, the last one shorter but not empty
            assert n >= 1 and s >= 1 and (n - 1) * s < t <= n * s, (i, t, n, s)
            assert n <= -(-t // MIN_DECODE_TILES)
            # no split longer than the launch's share unless the cap forces it
            assert s <= max(share, -(-t // cap)), (i, t, s, share, cap)
        assert ns + ns2 <= MAX_SPLITS and ns2 <= MAX_RING_SPLITS
        if ns + ns2 > 1:
            assert p["part0"][i] == part
            part += ns + ns2
        else:
            assert p["part0"][i] == -1
    assert p["n_items"] == sum(p["n_splits"]) + sum(p["n_splits2"])
    return p


def test_decode_short_rows_are_one_cta():
    p = check_decode(152, 32, 8, 128, 0, GLOBAL, [0, 1, 63, 64, 511])
    assert p["n_splits"] == [1] * 5 and p["part0"] == [-1] * 5
    assert p["split_tiles"] == [1, 1, 1, 2, 8]
    # a sliding layer reads at most its R ring slots whatever the position
    p = check_decode(152, 32, 8, 128, 512, SLIDING, [100, 511, 5000, 30000])
    assert p["n_splits"] == [1] * 4 and p["split_tiles"] == [2, 8, 8, 8]


def test_decode_one_long_row_fills_the_device():
    # 512 tiles would make 64 splits of 8 tiles: the cap leaves 32 of 16
    p = check_decode(152, 32, 8, 128, 0, GLOBAL, [32767])
    assert p["n_splits"] == [MAX_SPLITS] and p["split_tiles"] == [16]
    # 40 tiles: five splits of the minimum share
    p = check_decode(152, 32, 8, 128, 0, GLOBAL, [40 * TILE - 1])
    assert p["n_splits"] == [5] and p["split_tiles"] == [8] and p["part0"] == [0]


def test_decode_long_rows_capped_at_max_splits():
    p = check_decode(152, 8, 1, 64, 0, GLOBAL, [100000])
    assert p["n_splits"] == [MAX_SPLITS]
    assert p["split_tiles"] == [-(-tiles(100001) // MAX_SPLITS)]


def test_decode_hybrid_ring_is_its_own_segment():
    p = check_decode(152, 64, 8, 128, 512, FULL, [20000, 3, 511, 600])
    assert p["n_splits2"][1] == 1 and p["split_tiles2"][1] == 1
    assert all(n >= 1 for n in p["n_splits2"])
    assert p["split_tiles2"][2] == 8 and p["split_tiles2"][3] == 8
    q = check_decode(152, 64, 8, 128, 512, LOCAL, [20000, 3, 511, 600])
    assert q == p          # the same keys: the local layer reads its group's cache


def test_decode_more_keys_per_launch_gives_longer_splits():
    few = check_decode(152, 32, 8, 128, 0, GLOBAL, [16383] * 4)
    many = check_decode(152, 32, 8, 128, 0, GLOBAL, [16383] * 256)
    assert few["split_tiles"][0] < many["split_tiles"][0]
    assert few["n_splits"][0] > many["n_splits"][0]
    # a smaller device: fewer CTAs wanted, longer splits
    small = check_decode(16, 32, 8, 128, 0, GLOBAL, [16383] * 4)
    assert small["split_tiles"][0] > few["split_tiles"][0]


def test_decode_random_batches():
    rng = np.random.default_rng(7)
    for _ in range(300):
        kind = int(rng.integers(0, 4))
        Hk = int(rng.choice([1, 2, 4, 8, 16]))
        rep = int(rng.choice([1, 2, 4, 8, 16]))
        R = int(rng.integers(1, 4096))
        n = int(rng.integers(0, 513))
        hi = int(rng.choice([64, 2048, 40000, 2**20 - 1]))
        pos = [int(x) for x in rng.integers(0, hi, size=n)]
        num_sms = int(rng.choice([1, 8, 148, 152]))
        check_decode(num_sms, Hk * rep, Hk, int(rng.choice([64, 128])), R, kind, pos)


def test_decode_rejects_bad_shapes_and_rows():
    for args in [(0, 8, 2, 64, 0, GLOBAL), (152, 6, 4, 64, 0, GLOBAL),
                 (152, 8, 2, 96, 0, GLOBAL), (152, 8, 2, 64, 0, SLIDING),
                 (152, 8, 2, 64, 16, 4), (152, 64, 2, 64, 0, GLOBAL)]:
        with pytest.raises(KVError):
            kvi.plan_decode(*args, [5])
    for pos in ([-1], [2**20], [1] * 513):
        with pytest.raises(KVError):
            kvi.plan_decode(152, 8, 2, 64, 0, GLOBAL, pos)
    assert kvi.plan_decode(152, 8, 2, 64, 0, GLOBAL, [])["n_items"] == 0


def key_tiles(kind, R, lens, n):
    """Tiles of a chunk row's key space: its storage segments in order, each padded to
    whole tiles (a global layer's cache holds the chunk's own keys)."""
    ring = tiles(min(lens, R)) + tiles(n)
    if kind == SLIDING:
        return ring
    return tiles(lens + n) + (ring if kind in (FULL, LOCAL) else 0)


def expected_kind(kind, Hq, Hk, D, n):
    """0: mma.sync (D = 128 rows under 64 query rows on global and sliding layers);
    tcgen05 otherwise, 1 with two query tiles per CTA (D = 128), 2 with one (D = 64)."""
    if D == 64:
        return 2
    return 1 if (kind in (FULL, LOCAL) or n * Hq // Hk >= 64) else 0


PER_CTA, PER_SM = {0: 64, 1: 256, 2: 128}, {0: 2, 1: 1, 2: 2}


def planned_splits(num_sms, Hq, Hk, D, R, kind, lens, n, min_per):
    """Splits per row of the documented rule at a minimum of min_per blocks per split:
    within each launch kind, rows are split only when the longest row outweighs the
    average load per SM, into at most 16 pieces of about max(min_per, half that load)."""
    rep = Hq // Hk
    blocks = [-(-key_tiles(kind, R, lens[i], n[i]) // 2) for i in range(len(lens))]
    ns_all = [1] * len(lens)
    for kd in range(3):
        sel = [i for i in range(len(lens)) if expected_kind(kind, Hq, Hk, D, n[i]) == kd]
        if not sel:
            continue
        work = sum(-(-n[i] * rep // PER_CTA[kd]) * Hk * blocks[i] for i in sel)
        cap = num_sms * PER_SM[kd]
        if max(blocks[i] for i in sel) <= -(-work // cap):
            continue
        per = max(min_per, -(-work // (2 * cap)))
        for i in sel:
            ns = min(MAX_PREFILL_SPLITS, -(-blocks[i] // per))
            if ns > 1:
                bs = -(-blocks[i] // ns)
                ns = -(-blocks[i] // bs)
            ns_all[i] = max(1, ns)
    return ns_all


def reserve_min_per(num_sms, Hq, Hk, D, R, kind, lens, n):
    """The smallest minimum split length (4, 8, 16, ...) whose splits fit the partial
    vectors a cache reserves (PART_VECS_PER_SM per SM), as the planner chooses it."""
    min_per = MIN_PREFILL_BLOCKS
    while True:
        ns = planned_splits(num_sms, Hq, Hk, D, R, kind, lens, n, min_per)
        vecs = sum(k * n[i] * Hq for i, k in enumerate(ns) if k > 1)
        if vecs <= PART_VECS_PER_SM * num_sms or max(ns, default=1) == 1:
            return min_per, ns
        min_per *= 2


def check_prefill(num_sms, Hq, Hk, D, R, kind, lens, n):
    p = kvi.plan_prefill(num_sms, Hq, Hk, D, R, kind, lens, n)
    rep = Hq // Hk
    rows = len(lens)
    by_row = {i: [] for i in range(rows)}
    for j, r in enumerate(p["row"]):
        by_row[r].append(j)
    # launch order: kind by kind, input order within a kind
    order = [(p["kind"][j], p["row"][j]) for j in range(len(p["row"]))]
    assert order == sorted(order)
    # the partials fit the reserve of a cache on this many SMs
    assert p["part_vecs"] <= PART_VECS_PER_SM * num_sms
    min_per, want_ns = reserve_min_per(num_sms, Hq, Hk, D, R, kind, lens, n)
    assert p["n_splits"] == want_ns
    # the split decision and the share bound of a launch kind
    per_cta, per_sm = PER_CTA, PER_SM
    blocks = [-(-key_tiles(kind, R, lens[i], n[i]) // 2) for i in range(rows)]
    spans = []
    for kd in range(3):
        sel = [i for i in range(rows) if expected_kind(kind, Hq, Hk, D, n[i]) == kd]
        if not sel:
            continue
        work = sum(-(-n[i] * rep // per_cta[kd]) * Hk * blocks[i] for i in sel)
        cap = num_sms * per_sm[kd]
        split_any = max(blocks[i] for i in sel) > -(-work // cap)
        share = max(min_per, -(-work // (2 * cap)))
        for i in sel:
            ns = p["n_splits"][i]
            if not split_any:
                assert ns == 1, i
            if ns > 1:
                # blocks per split (all but the last): no more than the launch's share
                # unless the cap on splits forces it
                bs = p["tile0"][by_row[i][1]] // 2
                assert bs <= max(share, -(-blocks[i] // MAX_PREFILL_SPLITS)), (i, bs, share)
            elif split_any:
                assert blocks[i] <= share, (i, blocks[i], share)
    vecs = 0
    for i in range(rows):
        js = by_row[i]
        ns = p["n_splits"][i]
        assert len(js) == ns and 1 <= ns <= MAX_PREFILL_SPLITS
        assert ns <= max(1, -(-blocks[i] // MIN_PREFILL_BLOCKS))
        assert {p["kind"][j] for j in js} == {expected_kind(kind, Hq, Hk, D, n[i])}
        t = key_tiles(kind, R, lens[i], n[i])
        t0 = [p["tile0"][j] for j in js]
        t1 = [p["tile1"][j] for j in js]
        # contiguous, 128-key aligned, non-empty pieces of [0, end)
        assert t0[0] == 0 and t1[-1] == INF and t0[1:] == t1[:-1]
        assert all(a % 2 == 0 and a < t for a in t0), (i, t0, t)
        assert all(a < b for a, b in zip(t0, t1))
        parts = [p["part"][j] for j in js]
        if ns == 1:
            assert parts == [-1]
        else:
            stride = Hk * n[i] * rep
            assert parts == [parts[0] + k * stride for k in range(ns)]
            spans.append((parts[0], parts[0] + ns * stride))
            vecs += ns * stride
    spans.sort()
    assert spans == [] or spans[0][0] == 0
    assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))   # disjoint, no gaps
    assert p["part_vecs"] == vecs
    return p


def test_prefill_kernel_choice():
    lens, n = [100, 100, 100, 100], [1, 15, 16, 64]
    p = check_prefill(152, 32, 8, 128, 0, GLOBAL, lens, n)       # rep 4: 64 rows from n = 16
    assert [p["kind"][p["row"].index(i)] for i in range(4)] == [0, 0, 1, 1]
    p = check_prefill(152, 32, 8, 64, 0, GLOBAL, lens, n)
    assert set(p["kind"]) == {2}
    p = check_prefill(152, 32, 8, 128, 64, FULL, lens, n)
    assert set(p["kind"]) == {1}


def test_prefill_equal_rows_are_not_split():
    p = check_prefill(152, 64, 8, 128, 0, GLOBAL, [8192] * 64, [64] * 64)
    assert p["n_splits"] == [1] * 64 and p["part_vecs"] == 0


def test_prefill_one_long_row_among_short_ones_is_split():
    lens = [30000] + [10] * 7
    n = [64] * 8
    p = check_prefill(152, 32, 8, 128, 0, GLOBAL, lens, n)
    assert p["n_splits"][0] == MAX_PREFILL_SPLITS and p["n_splits"][1:] == [1] * 7
    assert p["part_vecs"] == MAX_PREFILL_SPLITS * 8 * 64 * 4
    # a sliding layer's keys stop at its ring and chunk: 512 + 64 keys, 5 blocks, 3 + 2
    p = check_prefill(152, 32, 8, 128, 512, SLIDING, lens, n)
    assert p["n_splits"] == [2] + [1] * 7
    assert [p["tile0"][j] for j in range(len(p["row"])) if p["row"][j] == 0] == [0, 6]


def test_prefill_random_batches():
    rng = np.random.default_rng(11)
    for _ in range(300):
        kind = int(rng.integers(0, 4))
        Hk = int(rng.choice([1, 2, 4, 8]))
        rep = int(rng.choice([1, 2, 4, 8, 16]))
        R = int(rng.integers(1, 4096))
        rows = int(rng.integers(0, 700))
        hi = int(rng.choice([64, 4096, 100000]))
        lens = [int(x) for x in rng.integers(0, hi, size=rows)]
        n = [int(x) for x in rng.integers(1, 65, size=rows)]
        check_prefill(int(rng.choice([1, 16, 152])), Hk * rep, Hk, int(rng.choice([64, 128])),
                      R, kind, lens, n)


def test_prefill_rejects_bad_rows():
    for lens, n in (([5], [0]), ([5], [65]), ([-1], [3]), ([2**20 - 2], [3])):
        with pytest.raises(KVError):
            kvi.plan_prefill(152, 8, 2, 64, 0, GLOBAL, lens, n)
    with pytest.raises(KVError):
        kvi.plan_prefill(152, 8, 2, 64, 0, 7, [5], [3])
    p = kvi.plan_prefill(152, 8, 2, 64, 0, GLOBAL, [], [])
    assert p["row"] == [] and p["part_vecs"] == 0


def test_prefill_partials_fit_the_create_reserve():
    """kv_append allocates nothing: every sub-chunk's key-split partials fit the vectors a
    cache reserves at create, min(1024 x SMs, B x Hq x 64 x 16).  Shapes that would need
    more (few SMs, long rows among short ones, wide GQA groups) get longer splits, down
    to none."""
    # Both launch kinds of D = 128 splitting at once: 64-token rows (two 128-row tiles per
    # CTA) and 15-token rows (mma.sync) behind one row at the largest length.  The
    # load-balancing rule alone asks for 1.32 x the reserve of 152 SMs.
    lens = [(1 << 20) - 64] + [361816] * 147 + [527055] * 149
    n = [64] * 148 + [15] * 149
    natural = planned_splits(152, 8, 2, 128, 0, GLOBAL, lens, n, MIN_PREFILL_BLOCKS)
    vecs = sum(k * n[i] * 8 for i, k in enumerate(natural) if k > 1)
    assert vecs > 1.3 * PART_VECS_PER_SM * 152
    p = check_prefill(152, 8, 2, 128, 0, GLOBAL, lens, n)
    assert 0 < p["part_vecs"] <= PART_VECS_PER_SM * 152 and max(p["n_splits"]) > 1
    # random long/short row mixes on any SM count
    rng = np.random.default_rng(5)
    worst = 0
    for _ in range(400):
        num_sms = int(rng.choice([1, 2, 8, 16, 152, 4096]))
        Hk = int(rng.choice([1, 2, 4, 8, 16]))
        rep = int(rng.choice([1, 2, 4, 8, 16]))
        D = int(rng.choice([64, 128]))
        kind = int(rng.integers(0, 4))
        R = int(rng.integers(1, 1 << 20))
        rows = int(rng.integers(1, 513))
        n_long = int(rng.integers(1, rows + 1))
        lens = ([int(x) for x in rng.integers((1 << 20) - 2 ** 18, (1 << 20) - 64, n_long)]
                + [int(x) for x in rng.integers(0, 1 << int(rng.integers(1, 16)),
                                                rows - n_long)])
        n = [64 if rng.random() < 0.7 else int(rng.integers(1, 65)) for _ in range(rows)]
        p = check_prefill(num_sms, Hk * rep, Hk, D, R, kind, lens, n)
        reserve = min(PART_VECS_PER_SM * num_sms, rows * Hk * rep * 64 * MAX_PREFILL_SPLITS)
        assert p["part_vecs"] <= reserve
        worst = max(worst, p["part_vecs"] / (PART_VECS_PER_SM * num_sms))
    assert worst > 0.5       # the search reached the bound's neighbourhood
