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


@pytest.mark.parametrize("Hq,Hk", [(16, 4), (32, 8), (8, 8)])
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
    with pytest.raises(kvi.KVError):
        c.step_graph([q] * 3, [k] * 3, [k] * 3, [q] * 3)
    with pytest.raises(kvi.KVError):
        c.copy_rows(c, [0], [1])
    with pytest.raises(ValueError):
        c.export_row(0)
    assert c.lens == [10, 3]
