"""The CPU oracle against what the pages and the mathematics fix (no GPU).

Each pin is chosen so that a plausible slip in the oracle -- a dropped term, a
wrong sign or index, a transposed operand, an off-by-one window -- fails at
least one test.  None of them re-types the oracle's own loops.
"""
import math
import os
import random

import numpy as np
import pytest
from scipy.special import softmax

import oracle
import synth
from conftest import GOLDEN

BF16_ONE = 0x3F80


def _bf16(x):
    """bf16 bits of exactly-representable small floats (test helper for constants)."""
    a = np.asarray(x, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def _f(bits):
    return oracle.bf16_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ bf16 rounding

def test_bf16_round_to_nearest_even():
    # 1 + 2^-8 is exactly halfway between bf16 1.0 and 1.0078125 -> ties to even (1.0)
    assert int(oracle.f32_to_bf16(np.float32(1.0 + 2 ** -8))) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1.0078125 (odd mantissa) and 1.015625 -> rounds up
    assert int(oracle.f32_to_bf16(np.float32(1.0 + 3 * 2 ** -8))) == 0x3F82
    # just above halfway rounds up
    assert int(oracle.f32_to_bf16(np.float32(1.0 + 2 ** -8 + 2 ** -20))) == 0x3F81
    assert int(oracle.f32_to_bf16(np.float32(-2.0))) == 0xC000
    # every bf16 value is a fixed point
    vals = np.arange(0, 0x7F80, 97, dtype=np.uint16)
    back = oracle.f32_to_bf16(oracle.bf16_to_f32(vals))
    assert np.array_equal(back, vals)


# ------------------------------------------------------------------ RoPE

@pytest.mark.parametrize("D", [8, 64, 128])
def test_rope_position_zero_is_identity(D):
    # cos 0 = 1 and sin 0 = 0 make rope(x, 0) == x bit for bit
    rng = np.random.default_rng(1)
    x = _bf16(rng.standard_normal((5, D)).astype(np.float32))
    assert np.array_equal(oracle.rope_bf16(x, 0), x)


@pytest.mark.parametrize("D,theta", [(8, 1e4), (64, 1e4), (128, 5e5)])
def test_rope_unit_vectors_give_cos_and_sin(D, theta):
    """Rotating a unit vector isolates one frequency: e_i -> (cos, sin) at (i, i+D/2) and
    e_{i+D/2} -> (-sin, cos).  Pins the half-split pairing, both signs and theta^(-2i/D)."""
    half = D // 2
    for p in (1, 2, 7, 100, 4097):
        for i in range(half):
            ang = p * math.pow(theta, (-2 * i) / D)
            c = np.float32(math.cos(ang))
            s = np.float32(math.sin(ang))
            e = np.zeros(D, dtype=np.uint16)
            e[i] = BF16_ONE
            r = oracle.rope_bf16(e[None], p, theta)[0]
            assert r[i] == oracle.f32_to_bf16(c) and r[i + half] == oracle.f32_to_bf16(s)
            assert np.count_nonzero(_f(r)) <= 2  # the rest are +-0
            e = np.zeros(D, dtype=np.uint16)
            e[i + half] = BF16_ONE
            r = oracle.rope_bf16(e[None], p, theta)[0]
            assert r[i] == oracle.f32_to_bf16(-s) and r[i + half] == oracle.f32_to_bf16(c)


def test_rope_table_matches_closed_form():
    c, s = oracle.rope_table(50, 16, 1e4)
    for p in range(50):
        for i in range(8):
            ang = p * math.pow(1e4, (-2 * i) / 16)
            assert c[p, i] == np.float32(math.cos(ang))
            assert s[p, i] == np.float32(math.sin(ang))
    # frequency pair 0 turns one radian per position
    assert c[1, 0] == np.float32(math.cos(1.0)) and s[3, 0] == np.float32(math.sin(3.0))


def test_rope_is_a_rotation_complex_form():
    """Against the complex-number form of RoPE (z_i = x_i + i x_{i+D/2}, z * e^{i p theta_i})
    in double: equal up to the float/bf16 rounding of the oracle."""
    rng = np.random.default_rng(7)
    D = 64
    x = _bf16(rng.standard_normal((20, D)).astype(np.float32))
    xf = _f(x)
    pos = rng.integers(0, 30000, size=20)
    r = _f(oracle.rope_bf16(x, pos))
    freqs = 1e4 ** (-2 * np.arange(D // 2) / D)
    z = (xf[:, :D // 2] + 1j * xf[:, D // 2:]) * np.exp(1j * pos[:, None] * freqs[None])
    ref = np.concatenate([z.real, z.imag], axis=1)
    # one f32 rounding of two products and a sum, then one bf16 rounding
    assert np.all(np.abs(r - ref) <= 2 ** -8 * np.abs(ref) + 4e-6 * np.abs(xf).max())
    # rotations preserve the norm of each pair
    n_in = xf[:, :D // 2] ** 2 + xf[:, D // 2:] ** 2
    n_out = r[:, :D // 2] ** 2 + r[:, D // 2:] ** 2
    assert np.allclose(n_out, n_in, rtol=2e-2, atol=1e-5)


def test_rope_scores_depend_only_on_distance():
    """q_m . k_n depends on m - n only (relative position); shifting both positions by the
    same amount changes the score only by rounding."""
    rng = np.random.default_rng(3)
    D = 128
    q = _bf16(rng.standard_normal((1, D)).astype(np.float32))
    k = _bf16(rng.standard_normal((1, D)).astype(np.float32))
    for m, n, shift in [(10, 3, 1000), (500, 500, 77), (7000, 12, 31)]:
        a = float(_f(oracle.rope_bf16(q, m))[0] @ _f(oracle.rope_bf16(k, n))[0])
        b = float(_f(oracle.rope_bf16(q, m + shift))[0] @ _f(oracle.rope_bf16(k, n + shift))[0])
        assert abs(a - b) <= 0.05 * math.sqrt(D), (m, n, shift, a, b)


def test_rope_is_linear_for_power_of_two_scale():
    rng = np.random.default_rng(5)
    x = _bf16(rng.standard_normal((4, 32)).astype(np.float32))
    x2 = _bf16(_f(x).astype(np.float32) * 2.0)
    assert np.array_equal(_f(oracle.rope_bf16(x2, 123)), 2.0 * _f(oracle.rope_bf16(x, 123)))


# ------------------------------------------------------------------ masks

def _read_golden_mask():
    rows = {}
    meta = {}
    with open(os.path.join(GOLDEN, "lab07_offset_mask.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                qp, vals = line.split(":")
                rows[int(qp)] = [v == "T" for v in vals.split()]
            else:
                k, v = line.split()
                meta[k] = int(v)
    return meta, rows


def test_mask_worked_example_lab07():
    meta, rows = _read_golden_mask()
    pos, t_new = meta["pos"], meta["t_new"]
    for i in range(t_new):
        not_allowed = [not oracle.visible(pos + i, j) for j in range(pos + t_new)]
        assert not_allowed == rows[pos + i]


def test_mask_single_query_sees_every_cached_key():
    # tiny-llm kv_cache.py `causal_kwargs`: one new token may see every cached key
    for pos in (0, 1, 5, 63):
        assert all(oracle.visible(pos, j) for j in range(pos + 1))
        assert not oracle.visible(pos, pos + 1)


def test_mask_start_zero_is_standard_causal():
    # with nothing cached the offset mask is the usual lower-triangular causal mask
    T = 6
    m = np.array([[oracle.visible(i, j) for j in range(T)] for i in range(T)])
    assert np.array_equal(m, np.tril(np.ones((T, T), dtype=bool)))


def test_sliding_window_keeps_exactly_w_keys():
    # inkling PR: the scan starts at t0 = qpos - window + 1
    for W in (1, 2, 8, 13):
        for p in range(40):
            vis = [j for j in range(p + 1) if oracle.visible(p, j, W)]
            assert vis == list(range(max(0, p - W + 1), p + 1))


# ------------------------------------------------------------------ attention

def _attend_onehot_values(n_keys, qpos, W, Hq=2, Hk=1):
    """K = 0 makes every score equal, so the output is the mean of the visible values;
    one-hot values make that mean reveal the exact visible set."""
    D = max(8, n_keys + (n_keys % 2))
    q = np.zeros((len(qpos), Hq, D), dtype=np.uint16)
    q[..., 0] = BF16_ONE
    k = np.zeros((n_keys, Hk, D), dtype=np.uint16)
    v = np.zeros((n_keys, Hk, D), dtype=np.uint16)
    for j in range(n_keys):
        v[j, :, j] = BF16_ONE
    return oracle.attend(q, qpos, k, v, 0, Hq, Hk, W=W)


def test_attention_worked_example_lab07_visible_sets():
    meta, rows = _read_golden_mask()
    pos, t_new = meta["pos"], meta["t_new"]
    out = _attend_onehot_values(pos + t_new, [pos + i for i in range(t_new)], W=0)
    for i in range(t_new):
        allowed = [not b for b in rows[pos + i]]
        expect = np.array(allowed, dtype=np.float64) / sum(allowed)
        assert np.array_equal(out[i, 0, :pos + t_new], expect)


@pytest.mark.parametrize("W", [1, 3, 8])
def test_attention_window_visible_sets(W):
    n = 20
    out = _attend_onehot_values(n, list(range(n)), W=W)
    for p in range(n):
        lo = max(0, p - W + 1)
        expect = np.zeros(n)
        expect[lo:p + 1] = 1.0 / (p + 1 - lo)
        assert np.array_equal(out[p, 1, :n], expect)


def test_attention_first_token_and_window_one_return_v():
    rng = np.random.default_rng(11)
    D, Hq, Hk = 16, 4, 2
    n = 9
    q = _bf16(rng.standard_normal((n, Hq, D)).astype(np.float32))
    k = _bf16(rng.standard_normal((n, Hk, D)).astype(np.float32))
    v = _bf16(rng.standard_normal((n, Hk, D)).astype(np.float32))
    out0 = oracle.attend(q[:1], [0], k, v, 0, Hq, Hk)
    for h in range(Hq):
        assert np.array_equal(out0[0, h], _f(v[0, h // 2]))
    out1 = oracle.attend(q, list(range(n)), k, v, 0, Hq, Hk, W=1)
    for p in range(n):
        for h in range(Hq):
            assert np.array_equal(out1[p, h], _f(v[p, h // 2]))


def test_attention_gqa_groups_are_contiguous():
    """Head h reads kv head h // rep (tiny_agent/generate.py reshapes (B,H,C,D) to
    (B,Hk,rep*C,D)); constant values per kv head expose the grouping exactly."""
    rng = np.random.default_rng(2)
    D, Hq, Hk, n = 8, 6, 3, 5
    q = _bf16(rng.standard_normal((n, Hq, D)).astype(np.float32))
    k = _bf16(rng.standard_normal((n, Hk, D)).astype(np.float32))
    v = np.zeros((n, Hk, D), dtype=np.uint16)
    for g in range(Hk):
        v[:, g, :] = _bf16(np.float32(g + 1))
    out = oracle.attend(q, list(range(n)), k, v, 0, Hq, Hk)
    for h in range(Hq):
        assert np.allclose(out[:, h, :], h // 2 + 1, rtol=0, atol=1e-12)


def test_attention_matches_softmax_matmul_brute_force():
    """softmax(Q K^T / sqrt(D) + mask) V with scipy/numpy on the oracle's rotated bf16
    Q and K: the attention loop (scale, max subtraction, window, GQA) in matrix form."""
    rng = np.random.default_rng(4)
    for (D, Hq, Hk, n, W, base) in [(16, 4, 2, 12, 0, 0), (32, 8, 2, 30, 7, 0),
                                     (64, 2, 1, 25, 5, 10)]:
        rep = Hq // Hk
        q = _bf16(rng.standard_normal((n, Hq, D)).astype(np.float32))
        k = _bf16(rng.standard_normal((n, Hk, D)).astype(np.float32))
        v = _bf16(rng.standard_normal((n, Hk, D)).astype(np.float32))
        pos = np.arange(base, base + n)
        qpos = pos[W if W else 0:]
        out = oracle.attend(q[W if W else 0:], qpos, k, v, base, Hq, Hk, W=W)
        Qr = _f(oracle.rope_bf16(q, pos[:, None]))
        Kr = _f(oracle.rope_bf16(k, pos[:, None]))
        Vf = _f(v)
        for h in range(Hq):
            g = h // rep
            S = Qr[:, h, :] @ Kr[:, g, :].T / math.sqrt(D)
            allowed = pos[None, :] <= pos[:, None]
            if W:
                allowed &= (pos[:, None] - pos[None, :]) < W
            S = np.where(allowed, S, -np.inf)
            ref = softmax(S, axis=1) @ Vf[:, g, :]
            got = out[:, h, :]
            assert np.allclose(got, ref[W if W else 0:], rtol=1e-12, atol=1e-12)


def test_attention_equal_keys_average_values():
    D, n = 8, 6
    rng = np.random.default_rng(8)
    q = _bf16(rng.standard_normal((1, 2, D)).astype(np.float32))
    k = np.repeat(_bf16(rng.standard_normal((1, 1, D)).astype(np.float32)), n, axis=0)
    v = _bf16(rng.standard_normal((n, 1, D)).astype(np.float32))
    # pre-RoPE keys that are equal stop being equal once rotated to different positions;
    # the zero key is the one key that every rotation leaves equal
    k[:] = 0
    out = oracle.attend(q, [n - 1], k, v, 0, 2, 1)
    assert np.allclose(out[0, 0], _f(v[:, 0]).mean(axis=0), rtol=0, atol=1e-15)


def test_attention_rejects_short_history():
    q = np.zeros((1, 2, 8), dtype=np.uint16)
    k = np.zeros((4, 1, 8), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.attend(q, [9], k, k, 0, 2, 1)           # history ends at position 3
    with pytest.raises(ValueError):
        oracle.attend(q, [9], k, k, 6, 2, 1, W=5)       # window starts at 5 < k_base 6
    oracle.attend(q, [9], k, k, 6, 2, 1, W=4)           # window [6, 9] is covered


# ------------------------------------------------------------------ ring slots

def _simulate_ring(chunks, W):
    """tiny_agent/generate.py `_append_chunk`: keep = pos >= new_lens - W,
    slot = pos % W, lpos[slot] = pos; applied chunk by chunk."""
    lpos = [-1] * W
    lens = 0
    for n in chunks:
        new_lens = lens + n
        for i in range(n):
            pos = lens + i
            if pos >= new_lens - W:
                lpos[pos % W] = pos
        lens = new_lens
    return lens, lpos


def _simulate_ring_inkling(chunks, W):
    """inkling PR: append after scoring, skipping s0 = max(0, S - win) rows of the batch."""
    ring = [-1] * W
    lens = 0
    for S in chunks:
        for s in range(max(0, S - W), S):
            ring[(lens + s) % W] = lens + s
        lens += S
    return lens, ring


def test_ring_slots_exhaustive_small():
    rnd = random.Random(0)
    for W in range(1, 9):
        for total in range(0, 41):
            for _ in range(6):
                chunks = []
                left = total
                while left > 0:
                    n = rnd.randint(1, min(20, left))
                    chunks.append(n)
                    left -= n
                lens, lpos = _simulate_ring(chunks, W)
                lens2, ring2 = _simulate_ring_inkling(chunks, W)
                expect = list(oracle.ring_positions(lens, W))
                assert lens == total == lens2
                assert lpos == expect == ring2, (W, chunks)


# ------------------------------------------------------------------ memory

def test_cache_bytes_lab07_answer():
    meta = {}
    with open(os.path.join(GOLDEN, "lab07_cache_bytes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                meta[k] = int(v)
    got = oracle.kv_nbytes(meta["batch"], meta["positions"], 0, meta["head_dim"],
                           meta["elem_bytes"], meta["layers"], meta["kv_heads"], 0, 0, 0)
    assert got == meta["bytes"] == 98304


def test_cache_bytes_inkling_memory_table():
    meta, table = {}, []
    with open(os.path.join(GOLDEN, "inkling_memory_table.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if len(parts) == 4:
                table.append(tuple(float(x) for x in parts))
            else:
                meta[parts[0]] = int(parts[1])
    GiB = 2 ** 30
    for ctx, full, ring, factor in table:
        ctx = int(ctx)
        args = (1, ctx, 0, meta["head_dim"], meta["elem_bytes"], meta["layers_global"],
                meta["kv_heads_global"], meta["layers_sliding"], meta["kv_heads_sliding"], 0)
        f_bytes = oracle.kv_nbytes(*args)
        r_bytes = oracle.kv_nbytes(1, ctx, meta["window"], *args[3:])
        # the page rounds half up to the printed precision
        assert abs(f_bytes / GiB - full) <= (0.05 if full < 100 else 0.5) + 1e-9
        assert abs(r_bytes / GiB - ring) <= 0.05 + 1e-9
        assert abs(f_bytes / r_bytes - factor) <= 0.05 + 1e-9
    per_full = oracle.kv_nbytes(1, 1, 0, 128, 4, 11, 8, 55, 16, 0)
    assert per_full == meta["per_token_full_KiB"] * 1024
    per_ring_growth = oracle.kv_nbytes(1, 1, 0, 128, 4, 11, 8, 0, 0, 0)
    assert per_ring_growth == meta["per_token_ring_KiB"] * 1024
    flat = oracle.kv_nbytes(1, 10 ** 6, meta["window"], 128, 4, 0, 0, 55, 16, 0)
    assert flat == meta["sliding_flat_MiB"] * 2 ** 20


# ------------------------------------------------------------------ stateless invariants

def test_oracle_chunking_and_incremental_are_the_same_call():
    """The oracle keeps no cache: answering queries in chunks 5+5+5+2 or one at a time gives
    the one-pass result bit for bit (Lab 07 section 3; test contract of section 2)."""
    seed, D, Hq, Hk = 9, 64, 4, 2
    n = 17
    q = synth.normal_bf16(seed, synth.Q, 0, 0, 0, range(n), Hq, D)
    k = synth.normal_bf16(seed, synth.K, 0, 0, 0, range(n), Hk, D)
    v = synth.normal_bf16(seed, synth.V, 0, 0, 0, range(n), Hk, D)
    full = oracle.attend(q, np.arange(n), k, v, 0, Hq, Hk)
    parts, s = [], 0
    for c in (5, 5, 5, 2):
        parts.append(oracle.attend(q[s:s + c], np.arange(s, s + c), k[:s + c], v[:s + c], 0,
                                   Hq, Hk))
        s += c
    assert np.array_equal(np.concatenate(parts), full)


# ------------------------------------------------------------------ hybrid layer

def _rand_bf16(rng, shape):
    return _bf16(rng.standard_normal(shape).astype(np.float32))


def test_hybrid_same_keys_and_full_window_equal_plain_attention():
    """With the local keys and values equal to the global ones and a window covering
    every position, each key appears twice with the same score: the two softmax halves
    share the same normalisation, so the result is plain attention over the global set."""
    rng = np.random.default_rng(21)
    D, Hq, Hk, n = 16, 4, 2, 11
    q = _rand_bf16(rng, (n, Hq, D))
    k = _rand_bf16(rng, (n, Hk, D))
    v = _rand_bf16(rng, (n, Hk, D))
    pos = np.arange(n)
    got = oracle.attend_hybrid(q, pos, k, v, k, v, Hq, Hk, W=n)
    ref = oracle.attend(q, pos, k, v, 0, Hq, Hk)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_hybrid_reduces_to_each_branch_when_the_other_is_negligible():
    """Keys that score far below the others (about -60 logits) drop out of the softmax:
    hybrid = global-only attention when the local keys are pushed away, and = local
    window attention when the global keys are.  theta is huge and the queries' first pair
    is zero, so RoPE leaves the relevant dot products unrotated (only pair 0 has
    frequency 1)."""
    rng = np.random.default_rng(22)
    D, Hq, Hk, n, W = 16, 2, 1, 9, 3
    theta = 1e30
    q = _bf16(np.full((n, Hq, D), 1.0, np.float32))
    q[:, :, 0] = 0
    q[:, :, D // 2] = 0                       # pair 0 (elements 0 and D/2) carries nothing
    far = _bf16(np.full((n, Hk, D), -16.0, np.float32))   # score -16 * (D-2) / 4 = -56
    k = _rand_bf16(rng, (n, Hk, D))
    k[:] = _bf16(np.float32(0.0))
    vg = _rand_bf16(rng, (n, Hk, D))
    vl = _rand_bf16(rng, (n, Hk, D))
    pos = np.arange(n)
    g_only = oracle.attend_hybrid(q, pos, k, vg, far, vl, Hq, Hk, W=W, theta=theta)
    assert np.allclose(g_only, oracle.attend(q, pos, k, vg, 0, Hq, Hk, theta=theta),
                       rtol=0, atol=1e-20)
    l_only = oracle.attend_hybrid(q, pos, far, vg, k, vl, Hq, Hk, W=W, theta=theta)
    assert np.allclose(l_only, oracle.attend(q, pos, k, vl, 0, Hq, Hk, W=W, theta=theta),
                       rtol=0, atol=1e-20)


def test_hybrid_log_sum_exp_merge_of_the_two_sets():
    """One softmax over two disjoint key sets is the two per-set softmaxes merged by their
    partition functions: out = (Zg Og + Zl Ol) / (Zg + Zl), with Z = sum of exp(scores)
    computed here from the rotated keys (scipy), and Og, Ol from the plain oracle."""
    rng = np.random.default_rng(23)
    D, Hq, Hk, n, W = 32, 4, 2, 14, 5
    q = _rand_bf16(rng, (n, Hq, D))
    kg, vg, kl, vl = (_rand_bf16(rng, (n, Hk, D)) for _ in range(4))
    pos = np.arange(n)
    got = oracle.attend_hybrid(q, pos, kg, vg, kl, vl, Hq, Hk, W=W)
    Og = oracle.attend(q, pos, kg, vg, 0, Hq, Hk)
    Ol = oracle.attend(q, pos, kl, vl, 0, Hq, Hk, W=W)
    Qr = _f(oracle.rope_bf16(q, pos[:, None]))
    Kgr = _f(oracle.rope_bf16(kg, pos[:, None]))
    Klr = _f(oracle.rope_bf16(kl, pos[:, None]))
    for h in range(Hq):
        g = h // (Hq // Hk)
        for p in range(n):
            sg = Kgr[: p + 1, g] @ Qr[p, h] / math.sqrt(D)
            lo = max(0, p - W + 1)
            sl = Klr[lo: p + 1, g] @ Qr[p, h] / math.sqrt(D)
            m = max(sg.max(), sl.max())
            Zg, Zl = np.exp(sg - m).sum(), np.exp(sl - m).sum()
            ref = (Zg * Og[p, h] + Zl * Ol[p, h]) / (Zg + Zl)
            assert np.allclose(got[p, h], ref, rtol=1e-11, atol=1e-12)
