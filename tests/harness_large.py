"""Full-size scenarios: inputs generated on the device, outputs and state sampled.

The counter-based generator fixes every q/k/v value by (seed, tensor, layer, row, seq,
position, head, d), so the oracle regenerates exactly the history of the rows and
layers it samples; nothing of the GPU path is stored or reused as an expected value.
Long histories are regenerated with the generator's device form (synth.fill_torch: the
same integer arithmetic, bit-identical to the numpy form by
tests/test_synth.py::test_device_generator_matches_numpy), which is input generation,
not the library under test.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth
from harness import check_close, torch_to_bits


class LargeScenario:
    def __init__(self, B, max_len, Hq, Hk, D, W=0, kinds=(0,), seed=0, theta=1e4):
        import torch
        import kv_cache_incremental_gb300 as kvi
        self.cache = kvi.KVCache(B, max_len, Hq, Hk, D, W, list(kinds), theta, 0)
        self.B, self.max_len, self.Hq, self.Hk, self.D, self.W = B, max_len, Hq, Hk, D, W
        self.kinds, self.seed, self.theta = list(kinds), seed, theta
        self.lens = np.zeros(B, dtype=np.int64)
        self.seq = np.zeros(B, dtype=np.int64)
        self.dev = torch.device("cuda", 0)
        self.max_ratio = 0.0

    def _gen_device(self, layer, C):
        import torch
        B, Hq, Hk, D = self.B, self.Hq, self.Hk, self.D
        rows = torch.arange(B, dtype=torch.int32, device=self.dev)
        seqs = torch.from_numpy(self.seq.astype(np.int32)).to(self.dev)
        pos0 = torch.from_numpy(self.lens.astype(np.int32)).to(self.dev)
        out = []
        for t, H in ((synth.Q, Hq), (synth.K, Hk), (synth.V, Hk)):
            x = torch.empty((B, C, H, D), dtype=torch.bfloat16, device=self.dev)
            synth.fill_device(x.data_ptr(), self.seed, t, layer, rows.data_ptr(), seqs.data_ptr(),
                              pos0.data_ptr(), B, C, H, D,
                              torch.cuda.current_stream().cuda_stream)
            out.append(x)
        return out

    def step(self, n_new, C, resets=(), keep_layers=()):
        """One step over all rows; returns {layer: out tensor} for the layers in keep_layers."""
        import torch
        if len(resets):
            self.cache.reset([int(r) for r in resets])
            for r in resets:
                self.lens[r] = 0
                self.seq[r] += 1
        n_new = [int(x) for x in n_new]
        kept = {}
        for layer in range(len(self.kinds)):
            q, k, v = self._gen_device(layer, C)
            out = self.cache.append(layer, q, k, v, n_new)
            if layer in keep_layers:
                kept[layer] = out
        self.cache.advance(n_new)
        torch.cuda.synchronize()
        lens_before = self.lens.copy()
        self.lens += np.asarray(n_new)
        return kept, lens_before

    def fill_to(self, targets, C=64):
        targets = np.asarray(targets, dtype=np.int64)
        while (self.lens < targets).any():
            n = np.minimum(C, targets - self.lens)
            self.step(n, C)

    # ------------------------------------------------------------------ checks
    def hist(self, tensor, layer, b, s, lo, hi, H):
        """Generator values of positions [lo, hi) of row b, sequence s: uint16 [n][H][D]."""
        if hi - lo <= 2048:
            return synth.normal_bf16(self.seed, tensor, layer, b, s, np.arange(lo, hi), H,
                                     self.D)
        import torch
        x = torch.empty((1, hi - lo, H, self.D), dtype=torch.bfloat16, device=self.dev)
        synth.fill_torch(x, self.seed, tensor, layer, [b], [s], [lo])
        return torch_to_bits(x)[0]

    def check_outputs(self, out, layer, rows, n_new, lens_before):
        """Every output element of the sampled rows of one layer against the oracle."""
        bits = torch_to_bits(out)
        W = self.W if self.kinds[layer] == 1 else 0
        for b in rows:
            n = int(n_new[b])
            if n == 0:
                continue
            L = int(lens_before[b])
            lo = max(0, L - (W - 1)) if W else 0
            s = int(self.seq[b])
            q = synth.normal_bf16(self.seed, synth.Q, layer, b, s, np.arange(L, L + n), self.Hq,
                                  self.D)
            kh = self.hist(synth.K, layer, b, s, lo, L + n, self.Hk)
            vh = self.hist(synth.V, layer, b, s, lo, L + n, self.Hk)
            ref = oracle.attend(q, np.arange(L, L + n), kh, vh, lo, self.Hq, self.Hk, W=W,
                                theta=self.theta)
            r = check_close(bits[b, :n], ref, f"layer {layer} row {b} lens {L} n {n}")
            self.max_ratio = max(self.max_ratio, r)

    def check_state(self, rows, layers):
        """Cache contents of sampled rows and layers, lpos of all rows, lens: bit for bit."""
        assert self.cache.lens == [int(x) for x in self.lens]
        R = self.cache.R
        for layer in layers:
            K, V = self.cache.storage(layer)
            for b in rows:
                L = int(self.lens[b])
                if L == 0:
                    continue
                if self.kinds[layer] == 0:
                    pos = np.arange(L)
                    slots = pos
                else:
                    ring = oracle.ring_positions(L, R)
                    slots = np.nonzero(ring >= 0)[0]
                    pos = ring[slots]
                s = int(self.seq[b])
                kr = oracle.rope_bf16(synth.normal_bf16(self.seed, synth.K, layer, b, s, pos,
                                                        self.Hk, self.D), pos[:, None], self.theta)
                vv = synth.normal_bf16(self.seed, synth.V, layer, b, s, pos, self.Hk, self.D)
                got_k = torch_to_bits(K[b][:, slots.tolist()]).transpose(1, 0, 2)
                got_v = torch_to_bits(V[b][:, slots.tolist()]).transpose(1, 0, 2)
                assert np.array_equal(got_k, kr), f"layer {layer} row {b}: K differs"
                assert np.array_equal(got_v, vv), f"layer {layer} row {b}: V differs"
        lp = self.cache.lpos()
        if lp is not None:
            lpos = lp.cpu().numpy()
            for b in range(self.B):
                assert np.array_equal(lpos[b], oracle.ring_positions(int(self.lens[b]), R)), \
                    f"row {b}: lpos differs"
