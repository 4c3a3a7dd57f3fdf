"""GPU path against the oracle at the full sizes of the benchmark configurations.

The cache is filled through the library's own chunked prefill with device-generated
inputs; outputs of sampled rows (every head and element of them) are checked against
the oracle, and cache contents, ring slots, lpos and lens bit for bit.
"""
import numpy as np
import pytest

from harness_large import LargeScenario

pytestmark = pytest.mark.gpu


def test_config3_decode_bandwidth_full_size():
    """B=64, Hq=32, Hk=8, D=128, one global layer, max_len=8192, lens uniform in [1024, 8092],
    one new token per row per step (the bench's workload)."""
    rng = np.random.default_rng(3)
    sc = LargeScenario(B=64, max_len=8192, Hq=32, Hk=8, D=128, seed=33)
    targets = rng.integers(1024, 8093, size=64)
    targets[:2] = [8092, 1024]  # both ends of the range
    sc.fill_to(targets)
    sample = [0, 1] + sorted(rng.choice(np.arange(2, 64), size=6, replace=False).tolist())
    for step in range(3):
        kept, lens_before = sc.step([1] * 64, C=1, keep_layers=(0,))
        if step in (0, 2):
            sc.check_outputs(kept[0], 0, sample, [1] * 64, lens_before)
    sc.check_state(sample, [0])


def test_config4_long_context_mixed_layout():
    """12 layers (5 and 11 global, the rest sliding W=512), B=16, Hq=64, Hk=8, D=128,
    max_len=32768, lens uniform in [16384, 32768 - steps], single-token decode steps.

    The cache fill (64-token chunks) is sampled whole-chunk: all 64 query positions of a
    row on a sliding and a global layer, for each kind of launch the planner makes on the
    way -- rows of equal length in two-tile tcgen05 CTAs (the call at 16384), a row cut
    into key splits merged afterwards (late calls, when few rows are still filling), and
    a row's last partial chunk of 5 tokens (5 x 8 query rows: the mma.sync kernel)."""
    import torch
    import kv_cache_incremental_gb300 as kvi
    rng = np.random.default_rng(4)
    kinds = [1, 1, 1, 1, 1, 0, 1, 1, 1, 1, 1, 0]
    sc = LargeScenario(B=16, max_len=32768, Hq=64, Hk=8, D=128, W=512, kinds=kinds, seed=44)
    targets = rng.integers(16384, 32768 - 8, size=16)
    targets[2] = 16384 + 64 * 40 + 5          # its last fill chunk has 5 tokens
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sc.fill_to(np.minimum(targets, 16384))
    kept, lens_before = sc.step(np.minimum(64, targets - sc.lens).tolist(), C=64,
                                keep_layers=(0, 5))
    n_fill = (sc.lens - lens_before).tolist()
    sc.check_outputs(kept[5], 5, [3], n_fill, lens_before)
    sc.check_outputs(kept[0], 0, [3, 7], n_fill, lens_before)
    seen_split = seen_small = False
    while (sc.lens < targets).any():
        n = np.minimum(64, targets - sc.lens)
        act = np.nonzero(n > 0)[0]
        plan = kvi.plan_prefill(sms, 64, 8, 128, 0, 0, sc.lens[act].tolist(), n[act].tolist())
        split_rows = [int(act[i]) for i, k in enumerate(plan["n_splits"]) if k > 1]
        want_split = bool(split_rows) and not seen_split
        want_small = n[2] == 5 and not seen_small
        if not (want_split or want_small):
            sc.step(n.tolist(), C=64)
            continue
        kept, lens_before = sc.step(n.tolist(), C=64, keep_layers=(5, 6, 10, 11))
        if want_split:
            seen_split = True
            b = split_rows[0]
            sc.check_outputs(kept[5], 5, [b], n.tolist(), lens_before)
            sc.check_outputs(kept[6], 6, [b], n.tolist(), lens_before)
        if want_small:
            seen_small = True
            assert plan["kind"][plan["row"].index(int(np.nonzero(act == 2)[0][0]))] == 0
            sc.check_outputs(kept[11], 11, [2], n.tolist(), lens_before)
            sc.check_outputs(kept[10], 10, [2], n.tolist(), lens_before)
    assert seen_split and seen_small
    for step in range(2):
        kept, lens_before = sc.step([1] * 16, C=1, keep_layers=(0, 5, 6, 11))
        sc.check_outputs(kept[5], 5, [1, 9], [1] * 16, lens_before)
        sc.check_outputs(kept[11], 11, [4], [1] * 16, lens_before)
        sc.check_outputs(kept[0], 0, list(range(16)), [1] * 16, lens_before)
        sc.check_outputs(kept[6], 6, [2, 12], [1] * 16, lens_before)
    sc.check_state([1, 4], [5])
    sc.check_state(list(range(16)), [0, 10])


def test_config5_continuous_batch_mix():
    """B=128, 4 layers (1 and 3 global; 0 and 2 sliding W=1024), Hq=16, Hk=4, D=64,
    max_len=16384, lens uniform in [0, 12000]; each step a right-padded C=64 batch with
    n_new 40% 1, 30% 0, 30% uniform [2, 64], after resetting 5% of the rows."""
    rng = np.random.default_rng(5)
    kinds = [1, 0, 1, 0]
    B = 128
    sc = LargeScenario(B=B, max_len=16384, Hq=16, Hk=4, D=64, W=1024, kinds=kinds, seed=55)
    sc.fill_to(rng.integers(0, 12001, size=B))
    for step in range(20):
        resets = rng.choice(B, size=max(1, B // 20), replace=False)
        u = rng.random(B)
        n = np.where(u < 0.4, 1, np.where(u < 0.7, 0, rng.integers(2, 65, size=B)))
        kept, lens_before = sc.step(n.tolist(), C=64, resets=resets.tolist(),
                                    keep_layers=(0, 1, 2, 3))
        # sample: a reset row, a decode row, a chunk row, an idle row, plus random ones
        pick = [int(resets[0])]
        for cond in (n == 1, n > 1, n == 0):
            idx = np.nonzero(cond)[0]
            if len(idx):
                pick.append(int(rng.choice(idx)))
        pick += rng.choice(B, size=2, replace=False).tolist()
        if step % 3 == 0 or step == 19:
            for layer in (0, 1) if step % 2 == 0 else (2, 3):
                sc.check_outputs(kept[layer], layer, sorted(set(pick)), n, lens_before)
    sc.check_state(sorted(set(pick)), [0, 1, 2, 3])
    sc.check_state(rng.choice(B, size=12, replace=False).tolist(), [0, 1, 2, 3])
