"""Benchmark: decode-attention HBM bandwidth and tokens/s against the preallocated cache.

Default workload (one global layer): B=64 rows, Hq=32, Hk=8, D=128, max_len=8192,
per-row cache lengths drawn uniformly from [1024, 8192 - reserve] (seeded), one new
token per row per step.  The cache is filled through the library's own chunked
prefill (64-token chunks); inputs are seeded synthetic bf16 values (Irwin-Hall(12)
approximation of N(0,1)).  A step is kv_append (RoPE + append + split-K decode +
combine) plus kv_advance for all rows.  The K/V read per step (~1.2 GB) is far above
the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_bw|long_ctx]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the
path has no exchange step); value = all ranks' units / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn HBM GB/s (% of ~8 TB/s) and tokens/s at B=64, 1k-8k ctx"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    # one global layer, the metric's configuration
    "decode_bw": dict(B=64, Hq=32, Hk=8, D=128, max_len=8192, W=0, kinds=[0], lo=1024),
    # 12 layers, sliding W=512 except layers 5 and 11, long context
    "long_ctx": dict(B=16, Hq=64, Hk=8, D=128, max_len=32768, W=512,
                     kinds=[1, 1, 1, 1, 1, 0, 1, 1, 1, 1, 1, 0], lo=16384),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_bw", choices=sorted(WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def initial_lens(cfg, total_steps, seed):
    rng = np.random.default_rng(seed)
    hi = cfg["max_len"] - total_steps - 1
    return rng.integers(cfg["lo"], hi + 1, size=cfg["B"]).astype(np.int64)


def kv_bytes_per_step(cfg, lens):
    """Algorithmic bytes of one decode step over all layers: every visible cached K/V byte
    once per kv head, plus q/k/v in, the new K/V written and the output."""
    B, Hq, Hk, D = cfg["B"], cfg["Hq"], cfg["Hk"], cfg["D"]
    total = 0.0
    for kind in cfg["kinds"]:
        keys = np.minimum(lens + 1, cfg["W"]) if kind == 1 else lens + 1
        total += float(np.sum(2.0 * Hk * keys * D * 2))
        total += B * (Hq + 2 * Hk) * D * 2 + 2 * B * Hk * D * 2 + B * Hq * D * 2
    return total


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


def traffic_record(kernel_file):
    """ncu DRAM traffic per launch for the decode kernel, if the committed capture matches
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    src = os.path.join(ROOT, "kv_cache_incremental_gb300", "csrc", kernel_file)
    try:
        with open(path) as f:
            rec = json.load(f)
        with open(src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()[:16]
        return rec if rec.get("source_sha256_16") == digest else None
    except Exception:
        return None


# ---------------------------------------------------------------------------- CPU oracle leg

def oracle_sample(cfg, lens, seed, budget_s=20.0, max_rows=None):
    """Time the CPU oracle on whole rows of one decode step of the same workload (first
    layer kind), until about `budget_s` of oracle time has been spent.  Returns
    (GB/s-equivalent, tokens/s, rows, threads, seconds)."""
    import oracle
    import synth
    Hq, Hk, D, W = cfg["Hq"], cfg["Hk"], cfg["D"], cfg["W"]
    kind = cfg["kinds"][0]
    spent, rows, byts = 0.0, 0, 0.0
    for b in range(cfg["B"]):
        if spent >= budget_s or (max_rows and rows >= max_rows):
            break
        p = int(lens[b])
        lo = max(0, p - W + 1) if kind == 1 else 0
        kh = synth.normal_bf16(seed, synth.K, 0, b, 0, range(lo, p + 1), Hk, D)
        vh = synth.normal_bf16(seed, synth.V, 0, b, 0, range(lo, p + 1), Hk, D)
        q = synth.normal_bf16(seed, synth.Q, 0, b, 0, [p], Hq, D)
        t0 = time.perf_counter()
        oracle.attend(q, [p], kh, vh, lo, Hq, Hk, W=W if kind == 1 else 0)
        spent += time.perf_counter() - t0
        rows += 1
        byts += 2.0 * Hk * (p + 1 - lo) * D * 2 + (Hq + 2 * Hk) * D * 2 + Hq * D * 2
    return byts / spent / 1e9, rows / spent, rows, oracle.num_threads(), spent


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    cfg = WORKLOADS[args.workload]
    lens = initial_lens(cfg, 2 * (args.warmup + args.steps), args.seed)
    # each step: a bounded sample of rows of one decode step, sized to finish in seconds
    for _ in range(max(0, args.warmup)):
        oracle_sample(cfg, lens, args.seed, budget_s=0.5, max_rows=1)
    total_b, total_t, rows, thr = 0.0, 0.0, 0, 1
    for _ in range(args.steps):
        gbs, _, r, thr, t = oracle_sample(cfg, lens, args.seed, budget_s=1.0, max_rows=2)
        total_b += gbs * t * 1e9
        total_t += t
        rows += r
    value = total_b / total_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, **{k: cfg[k] for k in (
            "B", "Hq", "Hk", "D", "max_len")}},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": thr, "kind": "oracle",
                         "sample": f"{rows} row-decodes (all {cfg['Hq']} heads, full history) "
                                   f"of the workload's first layer over {args.steps} steps"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- GPU leg

def fill_cache(cache, cfg, lens_target, seed, stream):
    """Prefill every row to its target length through the library, 64 tokens per call."""
    import torch
    import synth
    B, Hq, Hk, D = cfg["B"], cfg["Hq"], cfg["Hk"], cfg["D"]
    C = 64
    dev = torch.device("cuda", torch.cuda.current_device())
    q = torch.empty((B, C, Hq, D), dtype=torch.bfloat16, device=dev)
    k = torch.empty((B, C, Hk, D), dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    out = torch.empty_like(q)
    rows = torch.arange(B, dtype=torch.int32, device=dev)
    seqs = torch.zeros(B, dtype=torch.int32, device=dev)
    lens = np.zeros(B, dtype=np.int64)
    while (lens < lens_target).any():
        n = np.minimum(C, lens_target - lens).astype(np.int32)
        pos0 = torch.from_numpy(lens.astype(np.int32)).to(dev)
        for layer in range(len(cfg["kinds"])):
            for t, (x, H) in zip((synth.Q, synth.K, synth.V), ((q, Hq), (k, Hk), (v, Hk))):
                synth.fill_device(x.data_ptr(), seed, t, layer, rows.data_ptr(), seqs.data_ptr(),
                                  pos0.data_ptr(), B, C, H, D, stream.cuda_stream)
            cache.append(layer, q, k, v, n.tolist(), out=out, stream=stream)
        cache.advance(n.tolist(), stream=stream)
        lens += n
    torch.cuda.synchronize()


def run_ours(args):
    import torch
    import kv_cache_incremental_gb300 as kvi
    import synth

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    cfg = WORKLOADS[args.workload]
    B, Hq, Hk, D = cfg["B"], cfg["Hq"], cfg["Hk"], cfg["D"]
    n_layers = len(cfg["kinds"])
    K, Wm = args.steps, max(3, args.warmup)
    total_steps = 2 * (K + Wm)
    lens0 = initial_lens(cfg, total_steps, args.seed + rank)
    stream = torch.cuda.current_stream()
    dev = torch.device("cuda", local_rank)

    cache = kvi.KVCache(B, cfg["max_len"], Hq, Hk, D, cfg["W"], cfg["kinds"], 1e4, local_rank)
    t_fill = time.perf_counter()
    fill_cache(cache, cfg, lens0, args.seed + rank, stream)
    t_fill = time.perf_counter() - t_fill

    # decode inputs for every step, generated on the device (positions lens + s)
    steps_in = Wm + K
    qs = torch.empty((steps_in, n_layers, B, 1, Hq, D), dtype=torch.bfloat16, device=dev)
    ks = torch.empty((steps_in, n_layers, B, 1, Hk, D), dtype=torch.bfloat16, device=dev)
    vs = torch.empty_like(ks)
    rows = torch.arange(B, dtype=torch.int32, device=dev)
    seqs = torch.zeros(B, dtype=torch.int32, device=dev)
    for s in range(steps_in):
        pos0 = torch.from_numpy((lens0 + s).astype(np.int32)).to(dev)
        for layer in range(n_layers):
            for t, x, H in ((synth.Q, qs, Hq), (synth.K, ks, Hk), (synth.V, vs, Hk)):
                synth.fill_device(x[s, layer].data_ptr(), args.seed + rank, t, layer,
                                  rows.data_ptr(), seqs.data_ptr(), pos0.data_ptr(), B, 1, H, D,
                                  stream.cuda_stream)
    out = torch.empty((B, 1, Hq, D), dtype=torch.bfloat16, device=dev)
    ones = [1] * B
    torch.cuda.synchronize()

    def step(s):
        for layer in range(n_layers):
            cache.append(layer, qs[s, layer], ks[s, layer], vs[s, layer], ones, out=out,
                         stream=stream)
        cache.advance(ones, stream=stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for s in range(Wm):
        step(s)
    torch.cuda.synchronize()
    alg_bytes = sum(kv_bytes_per_step(cfg, lens0 + Wm + s) for s in range(K))

    clocks = ClockSampler(local_rank)
    cache.profile(True)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(Wm, Wm + K):
        step(s)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    prof = {k: cache.profile_read(k, reset=True) for k in ("append", "decode", "combine", "state")}
    cache.profile(False)
    launches = sum(p["launches"] for p in prof.values())

    # ---- end to end through the host-buffer entry point (pinned host memory)
    lens_e = lens0 + Wm + K
    hq = torch.empty((K + Wm, n_layers, B, 1, Hq, D), dtype=torch.bfloat16).pin_memory()
    hk = torch.empty((K + Wm, n_layers, B, 1, Hk, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    gq = torch.empty_like(qs)
    gk = torch.empty_like(ks)
    gv = torch.empty_like(vs)
    for s in range(K + Wm):
        pos0 = torch.from_numpy((lens_e + s).astype(np.int32)).to(dev)
        for layer in range(n_layers):
            for t, x, H in ((synth.Q, gq, Hq), (synth.K, gk, Hk), (synth.V, gv, Hk)):
                synth.fill_device(x[s, layer].data_ptr(), args.seed + rank, t, layer,
                                  rows.data_ptr(), seqs.data_ptr(), pos0.data_ptr(), B, 1, H, D,
                                  stream.cuda_stream)
    hq.copy_(gq)
    hk.copy_(gk)
    hv.copy_(gv)
    del gq, gk, gv
    hout = torch.empty((B, 1, Hq, D), dtype=torch.bfloat16).pin_memory()

    def step_host(s):
        for layer in range(n_layers):
            cache.append_host(layer, hq[s, layer], hk[s, layer], hv[s, layer], ones, out=hout,
                              stream=stream)
        cache.advance(ones, stream=stream)

    for s in range(Wm):
        step_host(s)
    torch.cuda.synchronize()
    e_bytes = sum(kv_bytes_per_step(cfg, lens_e + Wm + s) for s in range(K))
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for s in range(Wm, Wm + K):
        step_host(s)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = e0.elapsed_time(e1)

    # ---- max over ranks
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms, ms_e2e], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, ms_e2e = float(t[0]), float(t[1])
        tb = torch.tensor([alg_bytes, e_bytes], dtype=torch.float64, device=dev)
        dist.all_reduce(tb, op=dist.ReduceOp.SUM)
        alg_bytes, e_bytes = float(tb[0]), float(tb[1])
    if rank != 0:
        return
    value = alg_bytes / (ms / 1e3) / 1e9
    tok_s = world * B * K / (ms / 1e3)
    peak, peak_kind = measured_peaks()
    dec = prof["decode"]
    achieved = dec["bytes"] / (dec["ms"] / 1e3) / 1e9 if dec["ms"] > 0 else None
    traffic = traffic_record("decode.cu")
    per_launch_bytes = dec["bytes"] / max(1, dec["launches"])
    roofline = {
        "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
        "frac": (achieved / peak) if achieved else None,
        "traffic": (traffic["dram_bytes_per_launch"] if traffic else None),
        "kernel": "decode_kernel<128,1> (split-K GQA decode)",
        "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)",
        "alg_bytes_per_launch": per_launch_bytes,
        "avg_launch_ms": dec["ms"] / max(1, dec["launches"]),
        "frac_of_nominal_8TBs": (achieved / NOMINAL_HBM_GBS) if achieved else None,
    }
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "Hq": Hq, "Hk": Hk, "D": D,
                   "max_len": cfg["max_len"], "layers": n_layers,
                   "window": cfg["W"] or None, "lens": f"U[{cfg['lo']}, {cfg['max_len'] - total_steps - 1}]",
                   "l2": "inputs larger than L2 (K/V read per step >> 129 MB)",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": tok_s,
        "frac_of_nominal_8TBs": value / NOMINAL_HBM_GBS,
        "roofline": roofline,
        "e2e": {"value": e_bytes / (ms_e2e / 1e3) / 1e9, "unit": "GB/s",
                "tokens_per_s": world * B * K / (ms_e2e / 1e3),
                "h2d_bytes_per_step": n_layers * B * (Hq + 2 * Hk) * D * 2,
                "d2h_bytes_per_step": n_layers * B * Hq * D * 2},
        "gpu_launches": launches,
        "launches_by_kernel": {k: p["launches"] for k, p in prof.items()},
        "clocks": clk,
        "fill_s": t_fill,
    }
    if world == 1 and not args.no_cpu_baseline:
        gbs, tps, r, thr, t = oracle_sample(cfg, lens0 + Wm + K, args.seed + rank, budget_s=15.0)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": thr, "kind": "oracle",
                                "tokens_per_s": tps,
                                "sample": f"{r} row-decodes of one step (all {Hq} heads over the "
                                          f"row's whole history), {t:.1f} s of oracle time"}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
