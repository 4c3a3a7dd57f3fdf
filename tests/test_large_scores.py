"""Parity when scores leave the N(0,1) range.

"Lab 07 -- KV cache and sampling", section 2, fixes the contract: the incremental outputs
equal those of the full forward.  Real models reach attention scores far beyond what
bf16 N(0,1) queries and keys give (score standard deviation 1 in natural units, ~1.44 in
the kernels' log2 units), so these cases multiply every query by an exact power of two
(q_scale: an exponent shift in bf16, the oracle gets the same bits).  At q_scale = 16
scores have a standard deviation of ~23 log2 units: running maxima move by tens of units
as the keys stream by, which drives every rescaling path -- the lazy rescale of the
tcgen05 prefill (O in tensor memory rescaled only when a row's maximum grows by more than
8 log2 units), the per-tile rescale of the mma.sync prefill, the decode kernel's online
softmax and its split merge, the prefill key-split merge.  Outputs must stay within
|err| <= 2e-3 + 1e-2 |ref| of the oracle, the cache state bit for bit.

The tcgen05 cases also prove on the host that the lazy-rescale branch runs: from the
exact scores (oracle RoPE, double products) and the kernel's key-tile order over the
planned key splits (kv_plan_prefill), some query row's first rescale event clears the
threshold by a margin no float rounding of the kernel can close, and every tile before
it stays clear of the threshold by the same margin -- so the kernel's warp holding that
row takes the branch.
"""
import numpy as np
import pytest

import oracle
import synth
from harness import Scenario

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634
RESCALE_LOG2 = 8.0   # the tcgen05 prefill's lazy-rescale threshold
MARGIN = 0.05        # log2 units; the kernel's fp32 scores are within ~1e-3 of these


def _num_sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


def certain_rescales(sc, layer, rows, n_new):
    """Query rows of the next chunk of `rows` (global layer `layer`) whose tcgen05 prefill
    entry takes the lazy-rescale branch with certainty (see the module docstring)."""
    import kv_cache_incremental_gb300 as kvi
    D, Hq, Hk, rep = sc.D, sc.Hq, sc.Hk, sc.Hq // sc.Hk
    lens = [sc.lens[b] for b in rows]
    plan = kvi.plan_prefill(_num_sms(), Hq, Hk, D, 0, 0, lens, list(n_new))
    found = 0
    for i, b in enumerate(rows):
        ents = [j for j, r in enumerate(plan["row"]) if r == i]
        if not ents or plan["kind"][ents[0]] == 0:
            continue                        # the mma.sync kernel has no lazy rescale
        L, n = lens[i], n_new[i]
        pos = np.arange(L + n)
        k = oracle.rope_bf16(sc.gen(synth.K, layer, b, pos, Hk), pos[:, None], sc.theta)
        q = oracle.rope_bf16(sc.gen(synth.Q, layer, b, np.arange(L, L + n), Hq),
                             np.arange(L, L + n)[:, None], sc.theta)
        kf = oracle.bf16_to_f32(k).astype(np.float64)          # [keys][Hk][D]
        qf = oracle.bf16_to_f32(q).astype(np.float64)          # [n][Hq][D]
        for t in range(n):
            p = L + t
            for h in range(Hq):
                s = kf[: p + 1, h // rep] @ qf[t, h] * (LOG2E / np.sqrt(D))
                for j in ents:
                    t0, t1 = plan["tile0"][j], min(plan["tile1"][j], -(-(p + 1) // 64))
                    m_used = None
                    for tile in range(t0, t1):
                        mt = s[64 * tile: 64 * tile + 64].max()
                        if m_used is None:
                            m_used = mt
                            continue
                        gap = mt - (m_used + RESCALE_LOG2)
                        if abs(gap) < MARGIN:
                            break                   # too close to call: no claim
                        if gap > 0:
                            found += 1
                            break
    return found


@pytest.mark.parametrize("D,Hq,Hk,n,what", [
    (64, 8, 2, 64, "tcgen05, one query tile per CTA"),
    (128, 32, 4, 64, "tcgen05, two query tiles per CTA"),
])
def test_tcgen05_prefill_lazy_rescale_taken_and_within_tolerance(D, Hq, Hk, n, what):
    sc = Scenario(B=3, max_len=4096, Hq=Hq, Hk=Hk, D=D, seed=81, q_scale=16)
    sc.step([64, 40, 7], C=64, check_state=True)
    sc.step([64, 64, 64], C=64, check_state=True)
    rows, nn = [0, 1, 2], [n, n, n]
    # long history for row 0, so it is key-split too
    while sc.lens[0] < 3000:
        sc.step([64, 0, 0], C=64, check=False)
    assert certain_rescales(sc, 0, rows, nn) > 0, what
    sc.step(nn, C=n, check_state=True)


def test_mma_sync_prefill_and_key_splits_with_large_scores():
    """D = 128 chunks under 64 query rows (mma.sync), one row long enough to be split."""
    sc = Scenario(B=4, max_len=6000, Hq=16, Hk=4, D=128, seed=82, q_scale=16)
    sc.step([64, 9, 3, 15], C=64, check=False)
    while sc.lens[0] < 5000:
        sc.step([64, 0, 0, 0], C=64, check=False)
    import kv_cache_incremental_gb300 as kvi
    plan = kvi.plan_prefill(_num_sms(), 16, 4, 128, 0, 0, [sc.lens[b] for b in range(4)],
                            [12, 5, 2, 15])
    assert plan["n_splits"][0] > 1 and set(plan["kind"]) == {0}
    sc.step([12, 5, 2, 15], C=15, check_state=True)
    sc.step([1, 1, 1, 1], check_state=True)


@pytest.mark.parametrize("q_scale", [4, 64])
def test_decode_splits_and_merge_with_large_scores(q_scale):
    """Decode rows split over many CTAs (D = 128, rows to 4k keys), merged by the last."""
    sc = Scenario(B=4, max_len=4300, Hq=32, Hk=8, D=128, seed=83, q_scale=q_scale)
    targets = [4200, 1500, 65, 1]
    while any(t > l for t, l in zip(targets, sc.lens)):
        sc.step([min(64, t - l) for t, l in zip(targets, sc.lens)], C=64, check=False)
    for _ in range(3):
        sc.step([1, 1, 1, 1], check_state=True)


def test_sliding_and_hybrid_layers_with_large_scores():
    """Ring and chunk-scratch segments (sliding), and the three-segment hybrid softmax."""
    sc = Scenario(B=3, max_len=600, Hq=16, Hk=4, D=64, W=100, kinds=[1, 0, 2, 3], seed=84,
                  q_scale=16)
    sc.step([64, 30, 5], C=64, check_state=True)
    for _ in range(4):
        sc.step([64, 64, 40], C=64, check_state=True)
    for _ in range(3):
        sc.step([1, 1, 1], check_state=True)


def test_d64_decode_and_continuous_mix_with_large_scores():
    sc = Scenario(B=6, max_len=3000, Hq=16, Hk=4, D=64, W=512, kinds=[1, 0], seed=85,
                  q_scale=32)
    rng = np.random.default_rng(85)
    sc.step([64] * 6, C=64, check=False)
    for step in range(6):
        u = rng.random(6)
        n = np.where(u < 0.4, 1, np.where(u < 0.7, 0, rng.integers(2, 65, size=6)))
        resets = [int(rng.integers(0, 6))] if step == 3 else ()
        sc.step([int(x) for x in n], C=64, resets=resets, check_state=True)
