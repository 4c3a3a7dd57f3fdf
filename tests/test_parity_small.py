"""GPU path against the oracle on small cases (every output, every step, full state).

Sizes are ones the oracle finishes in seconds but that still span several key
tiles, a ragged tail, multiple sub-chunks and ring wraps.
"""
import numpy as np
import pytest

import oracle
import synth
from harness import Scenario, bf16_bits_to_torch, check_close, torch_to_bits

pytestmark = pytest.mark.gpu


def test_device_generator_matches_numpy():
    import torch
    out = torch.empty((3, 5, 4, 64), dtype=torch.bfloat16, device="cuda")
    synth.fill_torch(out, 7, synth.K, 2, rows=[0, 5, 9], seqs=[0, 1, 2], pos0=[0, 100, 4000])
    got = torch_to_bits(out)
    for i, (r, s, p0) in enumerate([(0, 0, 0), (5, 1, 100), (9, 2, 4000)]):
        ref = synth.normal_bf16(7, synth.K, 2, r, s, range(p0, p0 + 5), 4, 64)
        assert np.array_equal(got[i], ref)


def test_config1_tiny_chunked_prefill_then_decode():
    """1 global layer, B=2, Hq=4, Hk=2, D=64, max_len=128: row 0 prefills 17 tokens as
    chunks 5+5+5+2, row 1 prefills 9 in one chunk, then 8 single-token steps per row."""
    sc = Scenario(B=2, max_len=128, Hq=4, Hk=2, D=64, seed=1)
    sc.step([5, 9], C=9, check_state=True)
    sc.step([5, 0], C=5, check_state=True)
    sc.step([5, 0], C=5, check_state=True)
    sc.step([2, 0], C=2, check_state=True)
    for _ in range(8):
        sc.step([1, 1], C=1, check_state=True)
    assert sc.lens == [25, 17]


def test_chunked_prefill_equals_one_pass_bit_exact_cache():
    """Lab 07 section 3: 17 tokens as 5+5+5+2 give the one-pass result; the cache
    contents are identical bit for bit and the outputs agree within tolerance."""
    a = Scenario(B=1, max_len=64, Hq=4, Hk=2, D=64, seed=3)
    b = Scenario(B=1, max_len=64, Hq=4, Hk=2, D=64, seed=3)
    outs_a = []
    for n in (5, 5, 5, 2):
        outs_a.append(torch_to_bits(a.step([n], C=n)[0][1])[0, :n])
    out_b = torch_to_bits(b.step([17], C=17)[0][1])[0]
    Ka, Va = (torch_to_bits(x) for x in a.cache.storage(0))
    Kb, Vb = (torch_to_bits(x) for x in b.cache.storage(0))
    assert np.array_equal(Ka[:, :, :17], Kb[:, :, :17])
    assert np.array_equal(Va[:, :, :17], Vb[:, :, :17])
    got_a = oracle.bf16_to_f32(np.concatenate(outs_a)).astype(np.float64)
    check_close(out_b, got_a, "chunked vs one pass")
    a.check_state()
    b.check_state()


def test_config2_sliding_ring_wraps():
    """8 layers (layers 0-6 sliding W=8, layer 7 global), B=4, Hq=8, Hk=2, D=64,
    max_len=64: a 12+{0,3,5,7}-token prefill in one chunk (longer than the window),
    then 24 single-token decodes; the ring wraps 4+ times at different phases."""
    kinds = [1] * 7 + [0]
    sc = Scenario(B=4, max_len=64, Hq=8, Hk=2, D=64, W=8, kinds=kinds, seed=2)
    sc.step([12, 15, 17, 19], C=19, check_state=True)
    for _ in range(24):
        sc.step([1, 1, 1, 1], C=1, check_state=True)
    assert sc.lens == [36, 39, 41, 43]


@pytest.mark.parametrize("D,Hq,Hk", [(64, 4, 4), (64, 8, 4), (128, 16, 4), (128, 32, 4),
                                     (64, 16, 1), (128, 8, 8), (128, 32, 2)])
def test_head_layouts_decode_and_prefill(D, Hq, Hk):
    """GQA groups of 1, 2, 4, 8 and 16 query heads per kv head, both head dims."""
    sc = Scenario(B=3, max_len=300, Hq=Hq, Hk=Hk, D=D, W=40, kinds=[0, 1], seed=4)
    sc.step([70, 3, 130], C=130, check_state=True)   # several sub-chunks of 64
    for _ in range(3):
        sc.step([1, 1, 1], C=1)
    sc.step([1, 0, 20], C=20, check_state=True)      # mixed decode / chunk / idle


def test_long_decode_multi_split_and_tails():
    """Keys spanning many 64-key tiles so that split-K uses several splits per row."""
    sc = Scenario(B=3, max_len=3000, Hq=8, Hk=2, D=128, seed=5)
    sc.step([64, 64, 64], C=64)
    lens_target = [2900, 1000, 130]
    while max(t - l for t, l in zip(lens_target, sc.lens)) > 0:
        n = [min(64, max(0, t - l)) for t, l in zip(lens_target, sc.lens)]
        sc.step(n, C=64, check=False)
    sc.check_state()
    for _ in range(3):
        sc.step([1, 1, 1], C=1)


@pytest.mark.parametrize("D,Hq,Hk", [(64, 8, 2), (128, 16, 4)])
def test_one_token_sub_chunks(D, Hq, Hk):
    """Rows of 65 and 129 tokens end in a sub-chunk of one token, which takes the chunk path
    (append, prefill, ring commit), not the decode path; every layer kind, rings wrapping
    inside the chunk (W = 8)."""
    sc = Scenario(B=3, max_len=400, Hq=Hq, Hk=Hk, D=D, W=8, kinds=[1, 0, 2, 3], seed=12)
    sc.step([65, 129, 1], C=129, check_state=True)
    sc.step([1, 1, 1], C=1, check_state=True)
    sc.step([66, 0, 65], C=66, check_state=True)


def test_rows_subset_resets_and_idle_rows():
    sc = Scenario(B=6, max_len=200, Hq=4, Hk=2, D=64, W=16, kinds=[1, 0], seed=6)
    sc.step([10, 20, 0, 5], rows=[4, 0, 2, 5], C=20, check_state=True)
    sc.step([1, 1], rows=[0, 5], C=1, check_state=True)
    sc.step([3, 1, 30], rows=[5, 4, 1], C=30, resets=[4], check_state=True)
    sc.step([0, 0], rows=[1, 2], C=4, check_state=True)
    sc.step([17], rows=[3], C=17, resets=[3], check_state=True)


def test_padding_nan_never_leaks():
    """Pad tokens filled with NaN are routed to scratch and never reach a real output."""
    sc = Scenario(B=3, max_len=150, Hq=8, Hk=2, D=64, W=12, kinds=[1, 0], seed=7,
                  pad_value=0x7FC0)
    sc.step([5, 30, 1], C=33, check_state=True)
    sc.step([1, 2, 33], C=33, check_state=True)
    for _ in range(3):
        sc.step([1, 1, 1], C=4, check_state=True)


def test_window_one_and_window_at_least_max_len():
    a = Scenario(B=2, max_len=40, Hq=4, Hk=2, D=64, W=1, kinds=[1], seed=8)
    a.step([7, 3], C=7, check_state=True)
    a.step([1, 1], C=1, check_state=True)
    b = Scenario(B=2, max_len=40, Hq=4, Hk=2, D=64, W=64, kinds=[1, 0], seed=9)
    b.step([20, 5], C=20, check_state=True)
    b.step([1, 1], C=1, check_state=True)
    assert b.cache.R == 40  # W >= max_len: the ring holds every position (R = max_len)


def test_fill_to_max_len_and_full_rejection_changes_nothing():
    import kv_cache_incremental_gb300 as kvi
    import torch
    sc = Scenario(B=2, max_len=70, Hq=4, Hk=2, D=64, W=8, kinds=[0, 1], seed=10)
    sc.step([64, 10], C=64)
    sc.step([5, 1], C=5)
    before_k = [torch_to_bits(x) for x in sc.cache.storage(0)]
    q = torch.zeros((2, 2, 4, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((2, 2, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvi.KVCacheFull):
        sc.cache.append(0, q, k, k, [2, 1])   # 69 + 2 > 70
    with pytest.raises(kvi.KVCacheFull):
        sc.cache.advance([2, 1])
    torch.cuda.synchronize()
    after_k = [torch_to_bits(x) for x in sc.cache.storage(0)]
    assert all(np.array_equal(x, y) for x, y in zip(before_k, after_k))
    assert sc.cache.lens == [69, 11]
    sc.step([1, 1], C=1, check_state=True)   # exactly max_len
    assert sc.lens == [70, 12]


@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffer_entry_point_matches_device_entry_point(pinned):
    """kv_append_host with page-locked buffers (read and written by the kernels over the
    host link) and with pageable buffers (staged copies) gives kv_append's outputs."""
    import torch
    a = Scenario(B=2, max_len=100, Hq=8, Hk=2, D=128, W=10, kinds=[1, 0], seed=11)
    b = Scenario(B=2, max_len=100, Hq=8, Hk=2, D=128, W=10, kinds=[1, 0], seed=11)
    for n_new, C in (([20, 1], 20), ([1, 1], 1), ([3, 0], 4)):
        for layer in (0, 1):
            q, k, v = a.chunk_inputs(layer, [0, 1], n_new, C)
            out_dev = a.cache.append(layer, *(bf16_bits_to_torch(x, "cuda") for x in (q, k, v)),
                                     n_new)
            cpu = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) for x in (q, k, v)]
            out_host = torch.empty(cpu[0].shape, dtype=torch.bfloat16)
            if pinned:
                cpu = [x.pin_memory() for x in cpu]
                out_host = out_host.pin_memory()
            b.cache.append_host(layer, *cpu, n_new, out=out_host)
            torch.cuda.synchronize()
            d = torch_to_bits(out_dev)
            h = out_host.view(torch.int16).numpy().view(np.uint16)
            for i, n in enumerate(n_new):
                assert np.array_equal(d[i, :n], h[i, :n])
        for sc in (a, b):
            sc.cache.advance(n_new)
            sc.lens = [l + n for l, n in zip(sc.lens, n_new)]
    b.check_state()


def test_determinism_two_runs_bit_equal():
    outs = []
    for _ in range(2):
        sc = Scenario(B=3, max_len=400, Hq=8, Hk=2, D=64, W=24, kinds=[0, 1], seed=12)
        res = [torch_to_bits(o) for _, o in sc.step([100, 1, 37], C=100, check=False)]
        res += [torch_to_bits(o) for _, o in sc.step([1, 1, 1], C=1, check=False)]
        res += [torch_to_bits(x) for x in sc.cache.storage(0) + sc.cache.storage(1)]
        outs.append(res)
    for x, y in zip(*outs):
        assert np.array_equal(x, y)


def test_device_error_word_is_clear():
    sc = Scenario(B=2, max_len=100, Hq=4, Hk=2, D=64, seed=13)
    sc.step([30, 1], C=30)
    assert sc.cache.device_error() == 0
