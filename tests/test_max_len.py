"""The longest row a cache holds: max_len = 2^20 positions, the library's limit.

Row 0 takes the state of its first 2^20 - 10 tokens by import: the keys rotated by the
oracle's RoPE and the values, laid out as kv_export_row writes them (per layer K then V,
[Hk][positions][D]).  That is the state appending those tokens leaves, since every parity
test checks RoPE and append bit for bit.  Row 1 stays short.  A chunk of 8 tokens and two
decode tokens then fill row 0 to exactly max_len: RoPE at the last positions of the table,
a chunk row cut into key splits over 8192 128-key blocks, decode rows split 32 ways over
16384 64-key tiles.  Outputs are checked against the oracle, the cache's last positions
bit for bit, and one more token is refused without any change.
"""
import numpy as np
import pytest

import oracle
import synth
from harness import bf16_bits_to_torch, check_close, torch_to_bits

pytestmark = pytest.mark.gpu

MAX_LEN = 1 << 20
L0 = MAX_LEN - 10
SEED, HQ, HK, D = 41, 8, 1, 64


def stream(tensor, row, p0, p1, H):
    """Generator values of one stream at positions [p0, p1), in pieces to bound memory."""
    step = 1 << 16
    return np.concatenate([synth.normal_bf16(SEED, tensor, 0, row, 0,
                                             np.arange(s, min(p1, s + step)), H, D)
                           for s in range(p0, p1, step)])


def test_row_filled_to_max_len():
    import torch
    import kv_cache_incremental_gb300 as kvi
    dev = "cuda:0"
    cache = kvi.KVCache(2, MAX_LEN, HQ, HK, D, 0, [kvi.KV_GLOBAL])
    k0 = stream(synth.K, 0, 0, MAX_LEN, HK)            # row 0's whole history, pre-RoPE
    v0 = stream(synth.V, 0, 0, MAX_LEN, HK)
    k0_rot = oracle.rope_bf16(k0, np.arange(MAX_LEN)[:, None])
    flat = np.concatenate([k0_rot[:L0].transpose(1, 0, 2).ravel(),
                           v0[:L0].transpose(1, 0, 2).ravel()])
    assert flat.nbytes == 2 * HK * L0 * D * 2
    cache.import_row(0, bf16_bits_to_torch(flat, dev), keep=L0)
    assert cache.lens == [L0, 0]

    def inputs(C, n):
        """q, k, v (Bs = 2, C tokens) at the rows' current lengths; pads stay zero."""
        lens = cache.lens
        q = np.zeros((2, C, HQ, D), np.uint16)
        k = np.zeros((2, C, HK, D), np.uint16)
        v = np.zeros((2, C, HK, D), np.uint16)
        for b in range(2):
            p0, p1 = lens[b], lens[b] + n[b]
            if p1 > p0:
                q[b, :n[b]] = stream(synth.Q, b, p0, p1, HQ)
                k[b, :n[b]] = stream(synth.K, b, p0, p1, HK)
                v[b, :n[b]] = stream(synth.V, b, p0, p1, HK)
        return q, k, v

    def step(C, n):
        lens = cache.lens
        q, k, v = inputs(C, n)
        out = cache.append(0, *(bf16_bits_to_torch(x, dev) for x in (q, k, v)), n)
        cache.advance(n)
        torch.cuda.synchronize()
        got = torch_to_bits(out)
        for b in range(2):
            if n[b] == 0:
                continue
            pos = np.arange(lens[b], lens[b] + n[b])
            hk = k0 if b == 0 else stream(synth.K, 1, 0, pos[-1] + 1, HK)
            hv = v0 if b == 0 else stream(synth.V, 1, 0, pos[-1] + 1, HK)
            ref = oracle.attend(q[b, :n[b]], pos, hk[:pos[-1] + 1], hv[:pos[-1] + 1], 0, HQ, HK)
            check_close(got[b, :n[b]], ref, f"row {b} at {pos[0]}")

    step(8, [8, 5])                      # the chunk: row 0's 8 queries over ~2^20 keys
    step(1, [1, 1])                      # decode at 2^20 - 2
    step(1, [1, 1])                      # decode at 2^20 - 1: row 0 is full
    assert cache.lens == [MAX_LEN, 7]

    # the last positions of the cache, bit for bit (and a few imported ones)
    K, V = cache.storage(0)
    kb = torch_to_bits(K[0, :, MAX_LEN - 16:MAX_LEN])
    vb = torch_to_bits(V[0, :, MAX_LEN - 16:MAX_LEN])
    assert np.array_equal(kb, k0_rot[MAX_LEN - 16:].transpose(1, 0, 2))
    assert np.array_equal(vb, v0[MAX_LEN - 16:].transpose(1, 0, 2))
    assert np.array_equal(torch_to_bits(K[0, :, :16]), k0_rot[:16].transpose(1, 0, 2))

    # one more token for row 0 is refused, and nothing changes; row 1 goes on alone
    q, k, v = inputs(1, [1, 1])
    with pytest.raises(kvi.KVCacheFull):
        cache.append(0, *(bf16_bits_to_torch(x, dev) for x in (q, k, v)), [1, 1])
    torch.cuda.synchronize()
    assert cache.lens == [MAX_LEN, 7]
    assert np.array_equal(torch_to_bits(K[0, :, MAX_LEN - 16:MAX_LEN]), kb)
    step(1, [0, 1])
    assert cache.lens == [MAX_LEN, 8]
