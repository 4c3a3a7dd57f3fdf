"""Drive a KV-cache scenario through the C-ABI binding and check it against the oracle.

Inputs come from the counter-based generator (synth): the value of q/k/v at
(layer, row, seq, position, head, d) is fixed by the seed, so the oracle can
regenerate any row's whole history when it checks an output.  `seq` counts the
sequences a row has held (it advances on every reset).

Hybrid layers (kinds 2 = group's full layer, 3 = a local layer of the group): a layer's
own q/k/v streams feed its query and ring; the group's global keys and values are the
streams KG/VG of the group's full layer.

A row's history is a list of spans (p0, p1, seed, row, seq): positions p0 <= p < p1 came
from that stream.  A fresh or reset row has one open span of its own; a row that became a
prefix of another row (kv_copy_rows, kv_import_row) takes the source's spans up to the
kept length, then continues with a fresh stream of its own.

q_scale (a power of two) multiplies every query exactly (an exponent shift in bf16), so
scores leave the N(0,1) range by that factor: the oracle receives the same scaled bits.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth

TOL_ABS, TOL_REL = 2e-3, 1e-2  # |err| <= 2e-3 + 1e-2 |ref|, elementwise
_OPEN = 1 << 62                # end of a row's last history span


def bf16_bits_to_torch(bits, device):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def torch_to_bits(t):
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def check_close(got_bits, ref, what=""):
    got = oracle.bf16_to_f32(got_bits).astype(np.float64)
    err = np.abs(got - ref)
    bound = TOL_ABS + TOL_REL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; first at "
            f"{tuple(i)} got {got[tuple(i)]!r} ref {ref[tuple(i)]!r}; max err/bound "
            f"{float((err / bound).max()):.3f}")
    return float((err / bound).max()) if err.size else 0.0


class Scenario:
    """One cache plus the bookkeeping needed to regenerate every row's history."""

    def __init__(self, B, max_len, Hq, Hk, D, W=0, kinds=(0,), theta=1e4, seed=0, device=0,
                 pad_value=None, paged_blocks=None, q_scale=1):
        import kv_cache_incremental_gb300 as kvi
        self.kvi = kvi
        self.cache = kvi.KVCache(B, max_len, Hq, Hk, D, W, list(kinds), theta, device,
                                 paged_blocks=paged_blocks)
        self.B, self.max_len, self.Hq, self.Hk, self.D, self.W = B, max_len, Hq, Hk, D, W
        self.kinds = list(kinds)
        self.theta, self.seed = theta, seed
        self.dev = f"cuda:{device}"
        self.lens = [0] * B
        self.seq = [0] * B
        self.pad_value = pad_value  # None: generator values at pad positions; else a constant
        self.q_scale = q_scale
        assert q_scale > 0 and np.log2(q_scale) == np.round(np.log2(q_scale)), \
            "q_scale must be a power of two"
        self.spans = [[(0, _OPEN, seed, b, 0)] for b in range(B)]
        self.max_ratio = 0.0
        self.group, f = [], -1      # full layer of each hybrid layer's group, else -1
        for kind in self.kinds:
            f = len(self.group) if kind == 2 else f
            self.group.append(f if kind in (2, 3) else -1)

    # ------------------------------------------------------------------ inputs
    def gen(self, tensor, layer, row, positions, H):
        positions = np.asarray(positions, dtype=np.int64).reshape(-1)
        spans = self.spans[row]
        if len(spans) == 1:
            _, _, seed, srow, sseq = spans[0]
            x = synth.normal_bf16(seed, tensor, layer, srow, sseq, positions, H, self.D)
        else:
            x = np.empty((positions.size, H, self.D), np.uint16)
            for p0, p1, seed, srow, sseq in spans:
                m = (positions >= p0) & (positions < p1)
                if m.any():
                    x[m] = synth.normal_bf16(seed, tensor, layer, srow, sseq, positions[m], H,
                                             self.D)
        if tensor == synth.Q and self.q_scale != 1:
            x = oracle.f32_to_bf16(oracle.bf16_to_f32(x) * np.float32(self.q_scale))
        return x

    def _fresh_stream(self, b):
        """Row b starts a new sequence: a stream no earlier sequence of the row used."""
        self.seq[b] += 1
        return (self.seed, b, self.seq[b])

    def mark_reset(self, rows):
        """Bookkeeping of a kv_reset of `rows`: empty, each with a fresh stream."""
        for b in rows:
            self.lens[b] = 0
            seed, r, q = self._fresh_stream(b)
            self.spans[b] = [(0, _OPEN, seed, r, q)]

    def prefix_spans(self, b, keep):
        """Spans of row b's first `keep` positions."""
        return [(p0, min(p1, keep), seed, r, q) for p0, p1, seed, r, q in self.spans[b]
                if p0 < keep]

    def adopt(self, b, spans, keep):
        """Row b now holds `keep` positions from `spans` (a copy or an import): its history is
        those spans, then a fresh stream of its own from position keep on."""
        seed, r, q = self._fresh_stream(b)
        self.spans[b] = list(spans) + [(keep, _OPEN, seed, r, q)]
        self.lens[b] = keep

    def copy_rows(self, src, src_rows, dst_rows, keep=None):
        """kv_copy_rows from Scenario `src` (may be self) into this one, with the histories."""
        self.cache.copy_rows(src.cache, src_rows=list(src_rows), dst_rows=list(dst_rows),
                             keep=None if keep is None else list(keep))
        kept = [src.lens[s] if keep is None else k
                for s, k in zip(src_rows, keep or [None] * len(src_rows))]
        spans = [src.prefix_spans(s, k) for s, k in zip(src_rows, kept)]
        for d, sp, k in zip(dst_rows, spans, kept):
            self.adopt(d, sp, k)

    def import_row(self, row, buf, keep, src, src_row):
        """kv_import_row of a buffer exported from row src_row of Scenario `src`."""
        self.cache.import_row(row, buf, keep=keep)
        self.adopt(row, src.prefix_spans(src_row, keep), keep)

    def chunk_inputs(self, layer, rows, n_new, C):
        Bs = len(rows)
        q = np.zeros((Bs, C, self.Hq, self.D), np.uint16)
        k = np.zeros((Bs, C, self.Hk, self.D), np.uint16)
        v = np.zeros((Bs, C, self.Hk, self.D), np.uint16)
        for i, (b, n) in enumerate(zip(rows, n_new)):
            pos = np.arange(self.lens[b], self.lens[b] + C)
            q[i] = self.gen(synth.Q, layer, b, pos, self.Hq)
            k[i] = self.gen(synth.K, layer, b, pos, self.Hk)
            v[i] = self.gen(synth.V, layer, b, pos, self.Hk)
            if self.pad_value is not None and n < C:
                pad = np.uint16(self.pad_value)
                q[i, n:], k[i, n:], v[i, n:] = pad, pad, pad
        return q, k, v

    def global_inputs(self, layer, rows, n_new, C):
        """The group's global k, v of a hybrid layer's chunk (streams KG/VG of its full layer)."""
        f = self.group[layer]
        Bs = len(rows)
        kg = np.zeros((Bs, C, self.Hk, self.D), np.uint16)
        vg = np.zeros((Bs, C, self.Hk, self.D), np.uint16)
        for i, (b, n) in enumerate(zip(rows, n_new)):
            pos = np.arange(self.lens[b], self.lens[b] + C)
            kg[i] = self.gen(synth.KG, f, b, pos, self.Hk)
            vg[i] = self.gen(synth.VG, f, b, pos, self.Hk)
            if self.pad_value is not None and n < C:
                kg[i, n:] = vg[i, n:] = np.uint16(self.pad_value)
        return kg, vg

    def append_layer(self, layer, rows, rows_arg, n_new, C):
        """One layer's append through the binding; returns (q bits, out tensor)."""
        import torch
        q, k, v = self.chunk_inputs(layer, rows, n_new, C)
        qt, kt, vt = (bf16_bits_to_torch(x, self.dev) for x in (q, k, v))
        sentinel = torch.full_like(qt, 12345.0)
        kind = self.kinds[layer]
        if kind in (2, 3):
            kg = vg = None
            if kind == 2:
                kg, vg = (bf16_bits_to_torch(x, self.dev)
                          for x in self.global_inputs(layer, rows, n_new, C))
            out = self.cache.append_hybrid(layer, qt, kt, vt, list(n_new), k_global=kg,
                                           v_global=vg, rows=rows_arg, out=sentinel.clone())
        else:
            out = self.cache.append(layer, qt, kt, vt, list(n_new), rows_arg,
                                    out=sentinel.clone())
        return q, out

    # ------------------------------------------------------------------ one step
    def step(self, n_new, rows=None, C=None, resets=(), check=True, check_state=False):
        import torch
        rows_eff = list(range(len(n_new))) if rows is None else list(rows)
        if resets:
            self.cache.reset(list(resets))
            self.mark_reset(resets)
        C = C or max(1, max(n_new))
        outs = []
        for layer in range(len(self.kinds)):
            outs.append(self.append_layer(layer, rows_eff, rows, n_new, C))
        torch.cuda.synchronize()
        if check:
            for layer, (q, out) in enumerate(outs):
                self.check_outputs(layer, rows_eff, n_new, q, torch_to_bits(out))
        self.cache.advance(list(n_new), rows)
        for b, n in zip(rows_eff, n_new):
            self.lens[b] += n
        if check_state:
            self.check_state()
        return outs

    # ------------------------------------------------------------------ checks
    def check_outputs(self, layer, rows, n_new, q, out_bits):
        if self.kinds[layer] in (2, 3):
            return self.check_outputs_hybrid(layer, rows, n_new, q, out_bits)
        sliding = self.kinds[layer] == 1
        W = self.W if sliding else 0
        sentinel = np.uint16(0x4641)  # bf16(12345.0) rounds to 0x4641 (12352)
        for i, (b, n) in enumerate(zip(rows, n_new)):
            C = out_bits.shape[1]
            # padding positions and untouched rows keep the sentinel
            assert np.all(out_bits[i, n:] == sentinel), f"layer {layer} row {b}: pad written"
            if n == 0:
                continue
            L = self.lens[b]
            last = L + n - 1
            lo = max(0, L - (W - 1)) if W else 0
            hist = np.arange(lo, last + 1)
            kh = self.gen(synth.K, layer, b, hist, self.Hk)
            vh = self.gen(synth.V, layer, b, hist, self.Hk)
            ref = oracle.attend(q[i, :n], np.arange(L, L + n), kh, vh, lo, self.Hq, self.Hk, W=W,
                                theta=self.theta)
            r = check_close(out_bits[i, :n], ref, f"layer {layer} row {b} lens {L} n {n}")
            self.max_ratio = max(self.max_ratio, r)

    def check_outputs_hybrid(self, layer, rows, n_new, q, out_bits):
        sentinel = np.uint16(0x4641)
        f = self.group[layer]
        for i, (b, n) in enumerate(zip(rows, n_new)):
            assert np.all(out_bits[i, n:] == sentinel), f"layer {layer} row {b}: pad written"
            if n == 0:
                continue
            L = self.lens[b]
            hist = np.arange(L + n)
            kg = self.gen(synth.KG, f, b, hist, self.Hk)
            vg = self.gen(synth.VG, f, b, hist, self.Hk)
            kl = self.gen(synth.K, layer, b, hist, self.Hk)
            vl = self.gen(synth.V, layer, b, hist, self.Hk)
            ref = oracle.attend_hybrid(q[i, :n], np.arange(L, L + n), kg, vg, kl, vl, self.Hq,
                                       self.Hk, self.W, theta=self.theta)
            r = check_close(out_bits[i, :n], ref, f"hybrid layer {layer} row {b} lens {L} n {n}")
            self.max_ratio = max(self.max_ratio, r)

    def check_state(self):
        """Cache contents, ring slots, lpos and lens against the oracle, bit for bit."""
        import torch
        assert self.cache.lens == self.lens
        R = self.cache.R
        # (storage, layer of the streams, k stream, v stream, ring?) of every layer; a
        # hybrid layer has its group's cache and its own ring
        views = []
        for layer, kind in enumerate(self.kinds):
            if kind in (2, 3):
                views.append((self.cache.storage(layer), self.group[layer], synth.KG, synth.VG,
                              False))
                views.append((self.cache.ring_storage(layer), layer, synth.K, synth.V, True))
            else:
                views.append((self.cache.storage(layer), layer, synth.K, synth.V, kind == 1))
        for (K, V), layer, tk, tv, ringed in views:
            Kb, Vb = torch_to_bits(K), torch_to_bits(V)
            for b in range(self.B):
                L = self.lens[b]
                if L == 0:
                    continue
                if not ringed:
                    pos = np.arange(L)
                    slots = pos
                else:
                    ring = oracle.ring_positions(L, R)
                    slots = np.nonzero(ring >= 0)[0]
                    pos = ring[slots]
                kr = oracle.rope_bf16(self.gen(tk, layer, b, pos, self.Hk), pos[:, None],
                                      self.theta)
                vv = self.gen(tv, layer, b, pos, self.Hk)
                got_k = Kb[b][:, slots].transpose(1, 0, 2)
                got_v = Vb[b][:, slots].transpose(1, 0, 2)
                assert np.array_equal(got_k, kr), f"layer {layer} row {b}: K differs"
                assert np.array_equal(got_v, vv), f"layer {layer} row {b}: V differs"
        lp = self.cache.lpos()
        if lp is not None:
            lpos = lp.cpu().numpy()
            for b in range(self.B):
                assert np.array_equal(lpos[b], oracle.ring_positions(self.lens[b], R)), \
                    f"row {b}: lpos differs"
