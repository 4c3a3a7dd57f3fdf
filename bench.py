"""Benchmark: decode-attention HBM bandwidth and tokens/s against the preallocated cache.

Default workload (one global layer): B=64 rows, Hq=32, Hk=8, D=128, max_len=8192,
per-row cache lengths drawn uniformly from [1024, 8192 - reserve] (seeded), one new
token per row per step.  The cache is filled through the library's own chunked
prefill (64-token chunks); inputs are seeded synthetic bf16 values (Irwin-Hall(12)
approximation of N(0,1)).  A step is kv_append (RoPE + append + split-K decode +
combine) plus kv_advance for all rows.  The K/V read per step (~1.2 GB) is far above
the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_bw|long_ctx|hybrid|cont_batch]

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
# each workload's metric, the same in both arms (decode_bw: the headline metric above)
METRICS = {
    "decode_bw": METRIC,
    "long_ctx": "decode-attn HBM GB/s and tokens/s at B=16, 16k-32k ctx, 12 layers "
                "(10 sliding W=512, 2 global)",
    "hybrid": "decode-attn HBM GB/s and tokens/s at B=16, 16k-32k ctx, 3 hybrid groups of "
              "4 layers (W=512)",
    "cont_batch": "continuous-batch tokens/s (B=128, 4 layers, 64-token right-padded mix)",
}
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    # one global layer, the metric's configuration
    "decode_bw": dict(B=64, Hq=32, Hk=8, D=128, max_len=8192, W=0, kinds=[0], lo=1024,
                      steps=3000, per_round=100),
    # 12 layers, sliding W=512 except layers 5 and 11, long context
    "long_ctx": dict(B=16, Hq=64, Hk=8, D=128, max_len=32768, W=512,
                     kinds=[1, 1, 1, 1, 1, 0, 1, 1, 1, 1, 1, 0], lo=16384, steps=200,
                     per_round=20),
    # the long-context shapes as hybrid layers: 3 groups of 4 layers, each group sharing
    # one global K/V (written by its first layer), every layer with its own W=512 ring
    "hybrid": dict(B=16, Hq=64, Hk=8, D=128, max_len=32768, W=512,
                   kinds=[2, 3, 3, 3] * 3, lo=16384, steps=100, per_round=20),
    # continuous batching: 4 layers (1 and 3 global, 0 and 2 sliding W=1024), lens U[0, 12000];
    # each step resets 5% of the rows, then appends a right-padded 64-token batch with n_new
    # 1 (40%), 0 (30%) or U[2, 64] (30%)
    "cont_batch": dict(B=128, Hq=16, Hk=4, D=64, max_len=16384, W=1024, kinds=[1, 0, 1, 0],
                       lo=0, hi=12000, steps=50, per_round=50, mix=True),
}

HYBRID = (2, 3)  # KV_HYBRID_FULL, KV_HYBRID_LOCAL


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="0: the workload's default")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_bw", choices=sorted(WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-workloads", action="store_true",
                    help="the default workload's line without the long-context and "
                         "continuous-batch records")
    ap.add_argument("--fill-only", action="store_true",
                    help="time only the chunked-prefill cache fill of one cache (TFLOP/s)")
    ap.add_argument("--paged", action="store_true",
                    help="global layers in a paged cache (16-position blocks, a pool as large "
                         "as the dense cache)")
    ap.add_argument("--fill-to", type=int, default=0,
                    help="fill every row to this length instead of the workload's length "
                         "draw (small cases for profiling)")
    ap.add_argument("--max-len", type=int, default=0,
                    help="allocate the cache for this many positions instead of the "
                         "workload's (small cases for profiling; with --fill-to)")
    args = ap.parse_args(argv)
    if args.max_len:
        WORKLOADS[args.workload] = dict(WORKLOADS[args.workload], max_len=args.max_len)
    return args


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


def peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        return 1700.0


def initial_lens(cfg, total_steps, seed):
    rng = np.random.default_rng(seed)
    hi = cfg["max_len"] - total_steps - 1
    return rng.integers(cfg["lo"], hi + 1, size=cfg["B"]).astype(np.int64)


def decode_plan(cfg, args):
    """Timed steps K, warm-up steps, steps per cache fill, cache fills and the length reserve
    of a decode workload.  The configuration times per_round steps per cache fill; longer
    runs use several independently filled caches of that length (keeps the length
    distribution).  The reserve covers warm-up + timed steps, the same steps again with
    per-launch events (kernel durations), as decode-step graph replays, and end to end."""
    K = args.steps if args.steps else cfg["steps"]
    Wm = max(3, args.warmup)
    per_round = min(K, cfg["per_round"])
    rounds = (K + per_round - 1) // per_round
    return K, Wm, per_round, rounds, 4 * (Wm + per_round)


def decode_config(args, cfg, world):
    """`config` of a decode workload's JSON line, the same for both arms."""
    _, _, per_round, rounds, reserve = decode_plan(cfg, args)
    return {"workload": args.workload, "B": cfg["B"], "Hq": cfg["Hq"], "Hk": cfg["Hk"],
            "D": cfg["D"], "max_len": cfg["max_len"], "layers": len(cfg["kinds"]),
            "window": cfg["W"] or None,
            "lens": f"U[{cfg['lo']}, {cfg['max_len'] - reserve - 1}] per cache",
            "caches": rounds, "steps_per_cache": per_round, "paged": bool(args.paged),
            "l2": "inputs larger than L2 (K/V read per step >> 129 MB)",
            "parallelism": f"replicas x{world}"}


CONT_CHUNK = 64  # right-padded chunk width of the continuous-batch mix


def cont_config(args, cfg, world):
    """`config` of the continuous-batch workload's JSON line, the same for both arms."""
    return {"workload": args.workload, "B": cfg["B"], "Hq": cfg["Hq"], "Hk": cfg["Hk"],
            "D": cfg["D"], "max_len": cfg["max_len"], "layers": len(cfg["kinds"]),
            "window": cfg["W"], "lens": f"U[{cfg['lo']}, {cfg['hi']}] initial",
            "chunk": CONT_CHUNK,
            "mix": "n_new 1 (40%), 0 (30%), U[2,64] (30%); 5% of rows reset per step",
            "l2": "inputs larger than L2 (per step ~0.6 GB of K/V, 0.2 GB of inputs)",
            "parallelism": f"replicas x{world}"}


def kv_bytes_per_step(cfg, lens):
    """Algorithmic bytes of one decode step over all layers: every visible cached K/V byte
    once per kv head, plus q/k/v in, the new K/V written and the output."""
    B, Hq, Hk, D = cfg["B"], cfg["Hq"], cfg["Hk"], cfg["D"]
    total = 0.0
    for kind in cfg["kinds"]:
        local = np.minimum(lens + 1, cfg["W"])
        keys = local if kind == 1 else lens + 1 + local if kind in HYBRID else lens + 1
        total += float(np.sum(2.0 * Hk * keys * D * 2))
        # new key/value streams: one (global or sliding), a hybrid full layer's two, a
        # hybrid local layer's one (its ring's)
        kv_new = 2 if kind == 2 else 1
        total += B * (Hq + 2 * kv_new * Hk) * D * 2 + 2 * kv_new * B * Hk * D * 2 + B * Hq * D * 2
    return total


def append_layer(cache, kind, layer, q, k, v, kg, vg, n, out, stream):
    """One layer's append through the binding (hybrid layers with their global keys)."""
    if kind in HYBRID:
        return cache.append_hybrid(layer, q, k, v, n, k_global=kg if kind == 2 else None,
                                   v_global=vg if kind == 2 else None, out=out, stream=stream)
    return cache.append(layer, q, k, v, n, out=out, stream=stream)


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled DURING the timed region.

    Polls NVML (libnvidia-ml, read-only queries) from a thread every few ms; if NVML is
    not loadable, falls back to `nvidia-smi -lms`.  Samples are kept only between
    mark_start() and mark_stop()."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index, period_s=0.0005):
        import threading
        self.index, self.period = index, period_s
        self.samples = []  # (t, sm_mhz, max_mhz, reasons_mask)
        self.t0 = self.t1 = None
        self.stop_flag = threading.Event()
        self.thread = None
        self.nvml = None
        self.err = None

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByIndex failed")
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return lib, h, reasons_fn

    def _run(self):
        import ctypes
        lib, h, reasons_fn = self.nvml
        sm, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        # the maximum clock does not change: read once, then poll only the current clock and
        # the reasons (two queries per sample, so short regions get more samples)
        have_max = lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0
        while not self.stop_flag.is_set():
            t = time.perf_counter()
            ok = have_max and lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0  # SM clock
            ok = ok and reasons_fn(h, ctypes.byref(rs)) == 0
            if ok:
                self.samples.append((t, sm.value, mx.value, rs.value))
            self.stop_flag.wait(self.period)

    def start(self):
        import threading
        try:
            self.nvml = self._nvml_open()
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        except Exception as e:  # no NVML: nvidia-smi fallback
            self.err = f"nvml: {e}"
            self.thread = None
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index),
                     "--query-gpu=timestamp,clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                     "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception as e2:
                self.proc = None
                self.err += f"; nvidia-smi: {e2}"
        time.sleep(0.05)

    def mark_start(self):
        self.t0 = time.perf_counter()
        self.w0 = time.time()

    def mark_stop(self):
        self.t1 = time.perf_counter()
        self.w1 = time.time()

    def _smi_samples(self):
        import datetime
        proc = getattr(self, "proc", None)
        if proc is None:
            return
        proc.terminate()
        try:
            out, _ = proc.communicate(timeout=5)
        except Exception:
            proc.kill()
            out, _ = proc.communicate()
        bits = [0x8, 0x40, 0x20, 0x4]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                mask = sum(b for b, v in zip(bits, parts[3:7]) if v.lower().startswith("active"))
                # map wall-clock sample time into the perf_counter frame
                self.samples.append((self.t0 + (ts - self.w0), float(parts[1]), float(parts[2]),
                                     mask))
            except Exception:
                continue

    def stop(self):
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join(timeout=2)
        else:
            self._smi_samples()
        inside = [s for s in self.samples if self.t0 is not None and self.t0 <= s[0] <= self.t1]
        if not inside:
            return {"error": "no clock sample inside the timed region", "detail": self.err,
                    "samples_total": len(self.samples)}
        mask = 0
        for s in inside:
            mask |= s[3]
        return {"sm_mhz": float(np.median([s[1] for s in inside])),
                "sm_max_mhz": float(max(s[2] for s in inside)),
                "reasons": [name for bit, name in sorted(self.REASONS.items()) if mask & bit],
                "samples": len(inside), "source": "nvml" if self.thread is not None else "nvidia-smi"}


def traffic_record(kernel_file, workload):
    """ncu DRAM traffic per launch for the decode kernel, if the committed capture matches
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"decode_traffic_{workload}.json")
    src = os.path.join(ROOT, "kv_cache_incremental_gb300", "csrc", kernel_file)
    try:
        with open(path) as f:
            rec = json.load(f)
        with open(src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()[:16]
        return rec if rec.get("source_sha256_16") == digest else None
    except Exception:
        return None


HOLD_US = 1000  # blocking kernel before a device-timed region (see hold_stream)
START_NOTE = (f"device timing starts after a ~{HOLD_US} us blocking kernel queued behind the "
              "opening synchronize, so the first timed launches are already enqueued")


def hold_stream(stream, us=HOLD_US):
    """Keep `stream` busy for about `us` microseconds right before a device-timed region's
    start event (after the synchronize that opens it): by the time the start event executes,
    the host has already enqueued the first timed launches, so the region measures the device
    rather than the host's first enqueue (the blocking-kernel method of nvbench).  The kernel
    runs before the start event, outside the timed region; end-to-end regions do not use it."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * 2070))  # cycles at the maximum SM clock (2070 MHz)


def reduce_over_ranks(times, units, device):
    """Max over ranks of each time, sum over ranks of each unit count (replicas: the slowest
    rank bounds the whole job; every rank's work counts)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in times], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor([float(x) for x in units], dtype=torch.float64, device=device)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return t.tolist(), u.tolist()


# ---------------------------------------------------------------------------- CPU oracle leg

def oracle_sample(cfg, lens, seed, budget_s=20.0, max_rows=None):
    """Time the CPU oracle on whole rows of one decode step of the same workload (first
    layer kind), until about `budget_s` of oracle time has been spent or three times that
    in wall time (regenerating a row's history costs more than the oracle on it).  Returns
    (GB/s-equivalent, tokens/s, rows, threads, seconds of oracle time)."""
    import oracle
    import synth
    Hq, Hk, D, W = cfg["Hq"], cfg["Hk"], cfg["D"], cfg["W"]
    kind = cfg["kinds"][0]
    spent, rows, byts = 0.0, 0, 0.0
    wall0 = time.perf_counter()
    for b in range(cfg["B"]):
        if spent >= budget_s or (max_rows and rows >= max_rows) or \
                (rows and time.perf_counter() - wall0 >= 3 * budget_s):
            break
        p = int(lens[b])
        lo = max(0, p - W + 1) if kind == 1 else 0
        kh = synth.normal_bf16(seed, synth.K, 0, b, 0, range(lo, p + 1), Hk, D)
        vh = synth.normal_bf16(seed, synth.V, 0, b, 0, range(lo, p + 1), Hk, D)
        q = synth.normal_bf16(seed, synth.Q, 0, b, 0, [p], Hq, D)
        if kind in HYBRID:  # the group's global keys and the layer's local keys
            kg = synth.normal_bf16(seed, synth.KG, 0, b, 0, range(p + 1), Hk, D)
            vg = synth.normal_bf16(seed, synth.VG, 0, b, 0, range(p + 1), Hk, D)
            t0 = time.perf_counter()
            oracle.attend_hybrid(q, [p], kg, vg, kh, vh, Hq, Hk, W)
            spent += time.perf_counter() - t0
            keys = p + 1 + min(p + 1, W)
        else:
            t0 = time.perf_counter()
            oracle.attend(q, [p], kh, vh, lo, Hq, Hk, W=W if kind == 1 else 0)
            spent += time.perf_counter() - t0
            keys = p + 1 - lo
        rows += 1
        byts += 2.0 * Hk * keys * D * 2 + (Hq + 2 * Hk) * D * 2 + Hq * D * 2
    return byts / spent / 1e9, rows / spent, rows, oracle.num_threads(), spent


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    cfg = WORKLOADS[args.workload]
    config = decode_config(args, cfg, world)
    _, _, _, _, reserve = decode_plan(cfg, args)
    if not args.steps:
        args.steps = 10
    lens = initial_lens(cfg, reserve, args.seed)   # the first cache fill of the timed arm
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
        "impl": "reference", "metric": METRICS.get(args.workload, METRIC), "value": value,
        "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config,
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
    fill_cache_from(cache, cfg, np.zeros(cfg["B"], dtype=np.int64), lens_target, seed, stream)
    torch.cuda.synchronize()


def make_inputs(cfg, lens, n_steps, seed, dev, stream):
    """Decode inputs of n_steps steps for every layer, generated on the device at positions
    lens + s: tensors [n_steps, n_layers, B, 1, H, D] (q, k, v, and the global k, v of a
    hybrid full layer; those two are None without hybrid layers)."""
    import torch
    import synth
    B, Hq, Hk, D = cfg["B"], cfg["Hq"], cfg["Hk"], cfg["D"]
    L = len(cfg["kinds"])
    qs = torch.empty((n_steps, L, B, 1, Hq, D), dtype=torch.bfloat16, device=dev)
    ks = torch.empty((n_steps, L, B, 1, Hk, D), dtype=torch.bfloat16, device=dev)
    vs = torch.empty_like(ks)
    hyb = any(k in HYBRID for k in cfg["kinds"])
    kgs = torch.empty_like(ks) if hyb else None
    vgs = torch.empty_like(ks) if hyb else None
    rows = torch.arange(B, dtype=torch.int32, device=dev)
    seqs = torch.zeros(B, dtype=torch.int32, device=dev)
    for s in range(n_steps):
        pos0 = torch.from_numpy((lens + s).astype(np.int32)).to(dev)
        for layer in range(L):
            streams = [(synth.Q, qs, Hq), (synth.K, ks, Hk), (synth.V, vs, Hk)]
            if cfg["kinds"][layer] == 2:
                streams += [(synth.KG, kgs, Hk), (synth.VG, vgs, Hk)]
            for t, x, H in streams:
                synth.fill_device(x[s, layer].data_ptr(), seed, t, layer, rows.data_ptr(),
                                  seqs.data_ptr(), pos0.data_ptr(), B, 1, H, D,
                                  stream.cuda_stream)
    return qs, ks, vs, kgs, vgs


def step_inputs(inputs, s, layer):
    """(q, k, v, kg, vg) of one step and layer from make_inputs' tensors."""
    return tuple(None if x is None else x[s, layer] for x in inputs)


def run_fill_only(args):
    """Chunked-prefill throughput: fill one cache of the workload through kv_append in
    64-token chunks; the profiler range covers the last chunk call (all layers)."""
    import torch
    import kv_cache_incremental_gb300 as kvi
    cfg = WORKLOADS[args.workload]
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    B, Hq, Hk, D = cfg["B"], cfg["Hq"], cfg["Hk"], cfg["D"]
    pool = B * ((cfg["max_len"] + 15) // 16) if args.paged else None
    c = kvi.KVCache(B, cfg["max_len"], Hq, Hk, D, cfg["W"], cfg["kinds"], 1e4, 0,
                    paged_blocks=pool)
    if args.fill_to:
        target = np.full(B, args.fill_to, dtype=np.int64)
    else:
        target = initial_lens(cfg, 2 * (args.warmup + cfg["per_round"]), args.seed)
    c.profile(True)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    fill_cache(c, cfg, np.maximum(target - 64, 0), args.seed, stream)
    torch.cuda.profiler.start()
    fill_cache_from(c, cfg, np.maximum(target - 64, 0), target, args.seed, stream)
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    wall = time.perf_counter() - t0
    pre = c.profile_read("prefill", reset=True)
    app = c.profile_read("append", reset=True)
    com = c.profile_read("commit", reset=True)
    tflops = pre["flops"] / (pre["ms"] / 1e3) / 1e12 if pre["ms"] else None
    print(json.dumps({
        "metric": "chunked-prefill TFLOP/s (cache fill, 64-token chunks)", "value": tflops,
        "unit": "TFLOP/s", "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "Hq": Hq, "Hk": Hk, "D": D,
                   "layers": len(cfg["kinds"]), "fill_to": int(target.max()),
                   "paged": bool(args.paged)},
        "frac_of_bf16_sustained": tflops / peak_tflops() if tflops else None,
        "kernels": {"prefill": pre, "append": app, "commit": com}, "wall_s": wall,
        "flops_counted": "4*Hq*D per visible (query, key) pair, causal only"}), flush=True)


def fill_cache_from(cache, cfg, lens_from, lens_target, seed, stream):
    """Continue a fill from lens_from (the cache's current lengths) to lens_target."""
    import torch
    import synth
    B, Hq, Hk, D = cfg["B"], cfg["Hq"], cfg["Hk"], cfg["D"]
    C = 64
    dev = torch.device("cuda", torch.cuda.current_device())
    q = torch.empty((B, C, Hq, D), dtype=torch.bfloat16, device=dev)
    k = torch.empty((B, C, Hk, D), dtype=torch.bfloat16, device=dev)
    v, kg, vg = torch.empty_like(k), torch.empty_like(k), torch.empty_like(k)
    out = torch.empty_like(q)
    rows = torch.arange(B, dtype=torch.int32, device=dev)
    seqs = torch.zeros(B, dtype=torch.int32, device=dev)
    lens = lens_from.astype(np.int64).copy()
    while (lens < lens_target).any():
        n = np.minimum(C, lens_target - lens).astype(np.int32)
        pos0 = torch.from_numpy(lens.astype(np.int32)).to(dev)
        for layer, kind in enumerate(cfg["kinds"]):
            streams = [(synth.Q, q, Hq), (synth.K, k, Hk), (synth.V, v, Hk)]
            if kind == 2:
                streams += [(synth.KG, kg, Hk), (synth.VG, vg, Hk)]
            for t, x, H in streams:
                synth.fill_device(x.data_ptr(), seed, t, layer, rows.data_ptr(), seqs.data_ptr(),
                                  pos0.data_ptr(), B, C, H, D, stream.cuda_stream)
            append_layer(cache, kind, layer, q, k, v, kg, vg, n.tolist(), out, stream)
        cache.advance(n.tolist(), stream=stream)
        lens += n


def init_dist(local_rank, world):
    """One NCCL process group per job (the headline and its sub-workloads share it)."""
    import torch
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("nccl")


def step_times(events):
    """Per-step device times (ms) from events recorded after each step (events[0]: start)."""
    ms = [a.elapsed_time(b) for a, b in zip(events, events[1:])]
    if not ms:
        return None
    return {"first": ms[0], "median": float(np.median(ms)), "min": min(ms), "max": max(ms),
            "last": ms[-1], "n": len(ms)}


def run_ours(args, sub=False):
    """A decode workload; returns rank 0's JSON record (None on other ranks).  sub: a
    sub-record of the headline line (no CPU baseline)."""
    import torch
    import kv_cache_incremental_gb300 as kvi

    rank, local_rank, world = dist_env()
    init_dist(local_rank, world)
    cfg = WORKLOADS[args.workload]
    B, Hq, Hk, D = cfg["B"], cfg["Hq"], cfg["Hk"], cfg["D"]
    n_layers = len(cfg["kinds"])
    K, Wm, per_round, rounds, reserve = decode_plan(cfg, args)
    stream = torch.cuda.current_stream()
    dev = torch.device("cuda", local_rank)

    caches, lens0 = [], []
    t_fill = time.perf_counter()
    pre = {"launches": 0, "ms": 0.0, "bytes": 0.0, "flops": 0.0}
    for r in range(rounds):
        seed_r = args.seed + 7919 * rank + 104729 * r
        pool = B * ((cfg["max_len"] + 15) // 16) if args.paged else None
        c = kvi.KVCache(B, cfg["max_len"], Hq, Hk, D, cfg["W"], cfg["kinds"], 1e4, local_rank,
                        paged_blocks=pool)
        if args.fill_to:  # small-case profiling: every row at the same, shorter length
            l0 = np.full(B, min(args.fill_to, cfg["max_len"] - reserve - 1), dtype=np.int64)
        else:
            l0 = initial_lens(cfg, reserve, seed_r)
        c.profile(r == 0)  # the chunked-prefill kernel, timed on the first fill
        fill_cache(c, cfg, l0, seed_r, stream)
        if r == 0:
            pre = c.profile_read("prefill", reset=True)
            c.profile(False)
        caches.append((c, seed_r))
        lens0.append(l0)
    t_fill = time.perf_counter() - t_fill
    steps_in_round = [min(per_round, K - r * per_round) for r in range(rounds)]

    out = torch.empty((B, 1, Hq, D), dtype=torch.bfloat16, device=dev)
    ones = [1] * B

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- warm-up on cache 0, then the timed rounds (inputs generated beforehand)
    inputs = []
    for r in range(rounds):
        start = Wm if r == 0 else 0
        n = steps_in_round[r] + start
        inputs.append(make_inputs(cfg, lens0[r], n, caches[r][1], dev, stream))
    torch.cuda.synchronize()
    kinds = cfg["kinds"]
    hybrid = any(k in HYBRID for k in kinds)
    alg_bytes = 0.0
    for r in range(rounds):
        base = lens0[r] + (Wm if r == 0 else 0)
        alg_bytes += sum(kv_bytes_per_step(cfg, base + s) for s in range(steps_in_round[r]))

    def slices(inputs, first_of):
        """Per round, step and layer, the (q, k, v, kg, vg) views of that step's inputs,
        taken before a timed region so that it holds only library calls."""
        return [[[step_inputs(inputs[r], s, layer) for layer in range(n_layers)]
                 for s in range(first_of(r), first_of(r) + steps_in_round[r])]
                for r in range(rounds)]

    def run_rounds(first_of, after_step=None, after_layer=None, views=None):
        views = views or slices(inputs, first_of)
        for r in range(rounds):
            c = caches[r][0]
            for sv in views[r]:
                for layer in range(n_layers):
                    append_layer(c, kinds[layer], layer, *sv[layer], ones, out, stream)
                    if after_layer:
                        after_layer(c, kinds[layer])
                c.advance(ones, stream=stream)
                if after_step:
                    after_step()

    # Timed region: the workload alone.  The library's per-launch events (kernel
    # durations) cost ~10% of a 12-layer step, so they run in a second pass below; an
    # event after each step (a stream marker, no host wait) gives the per-step times.
    # The warm-up steps run right before it, after the clock sampler has started, so the
    # GPU is busy up to the first timed step.
    clocks = ClockSampler(local_rank)
    clocks.start()
    for s in range(Wm):
        for layer in range(n_layers):
            append_layer(caches[0][0], kinds[layer], layer, *step_inputs(inputs[0], s, layer),
                         ones, out, stream)
        caches[0][0].advance(ones, stream=stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    e0, e1 = evs[0], evs[-1]
    it = iter(evs[1:])
    timed_views = slices(inputs, lambda r: Wm if r == 0 else 0)
    hold_stream(stream)
    clocks.mark_start()
    torch.cuda.profiler.start()  # profilers started with --profile-from-start off see this range
    e0.record(stream)
    h0 = time.perf_counter()
    run_rounds(lambda r: Wm if r == 0 else 0, after_step=lambda: next(it).record(stream),
               views=timed_views)
    host_ms = (time.perf_counter() - h0) * 1e3   # enqueue time of the K steps
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    clocks.mark_stop()
    barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    per_step = step_times(evs)

    # Kernel durations: the same number of steps per cache, continuing from where the timed
    # region left each cache, with CUDA events around every library launch (on the launch
    # stream).
    inputs = []
    for r in range(rounds):
        lens_p = lens0[r] + (Wm if r == 0 else 0) + steps_in_round[r]
        inputs.append(make_inputs(cfg, lens_p, steps_in_round[r], caches[r][1] + 1, dev, stream))
    torch.cuda.synchronize()
    for c, _ in caches:
        c.profile(True)
    kkinds = ("append", "decode", "combine", "state")
    prof = {k: {"launches": 0, "ms": 0.0, "bytes": 0.0, "flops": 0.0} for k in kkinds}
    # the decode launches by layer kind (global, sliding, hybrid), read after every layer
    by_kind = {}

    def after_layer(c, kind):
        rec = c.profile_read("decode", reset=True)
        name = "global" if kind == 0 else "sliding" if kind == 1 else "hybrid"
        acc = by_kind.setdefault(name, {"launches": 0, "ms": 0.0, "bytes": 0.0})
        for f in acc:
            acc[f] += rec[f]
        for f in rec:
            prof["decode"][f] += rec[f]

    run_rounds(lambda r: 0, after_layer=after_layer)
    torch.cuda.synchronize()
    for c, _ in caches:
        for k in kkinds:
            rec = c.profile_read(k, reset=True)
            for f in rec:
                prof[k][f] += rec[f]
        c.profile(False)
    launches = sum(p["launches"] for p in prof.values())
    peak, peak_kind = measured_peaks()
    split = {name: {"launches": a["launches"], "avg_launch_ms": a["ms"] / max(1, a["launches"]),
                    "alg_bytes_per_launch": a["bytes"] / max(1, a["launches"]),
                    "achieved": a["bytes"] / (a["ms"] / 1e3) / 1e9 if a["ms"] else None,
                    "frac": a["bytes"] / (a["ms"] / 1e3) / 1e9 / peak if a["ms"] else None}
             for name, a in by_kind.items()}
    del inputs

    # ---- the same steps as decode-step graph replays (kv_step_graph: one graph launch per
    # step re-planned from the host lengths), each step pointed at its own inputs
    graph_bytes, inputs, graphs = 0.0, [], []
    outs_l = [torch.empty((B, 1, Hq, D), dtype=torch.bfloat16, device=dev)
              for _ in range(n_layers)]
    for r in range(rounds):
        lens_g = lens0[r] + (Wm if r == 0 else 0) + 2 * steps_in_round[r]
        qs, ks, vs, kgs, vgs = make_inputs(cfg, lens_g, steps_in_round[r], caches[r][1] + 2,
                                           dev, stream)
        inputs.append((qs, ks, vs, kgs, vgs))
        per_layer = lambda x, s: [x[s, l] for l in range(n_layers)]
        glob = lambda x, s: ([x[s, l] if kinds[l] == 2 else None for l in range(n_layers)]
                             if hybrid else None)
        g = caches[r][0].step_graph(per_layer(qs, 0), per_layer(ks, 0), per_layer(vs, 0), outs_l,
                                    k_global=glob(kgs, 0), v_global=glob(vgs, 0))
        bufs = [g.buffers(per_layer(qs, s), per_layer(ks, s), per_layer(vs, s), outs_l,
                          k_global=glob(kgs, s), v_global=glob(vgs, s))
                for s in range(steps_in_round[r])]
        graphs.append((g, bufs))
        graph_bytes += sum(kv_bytes_per_step(cfg, lens_g + s) for s in range(steps_in_round[r]))
    torch.cuda.synchronize()
    barrier()
    e0.record(stream)
    for g, bufs in graphs:
        for b in bufs:
            g.launch(stream, buffers=b)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_graph = e0.elapsed_time(e1) if graphs else None
    for g, _ in graphs:
        g.close()
    del inputs, graphs

    # ---- end to end through the host-buffer entry point (pinned host memory)
    e_bytes, ms_e2e = 0.0, 0.0
    hout = torch.empty((B, 1, Hq, D), dtype=torch.bfloat16).pin_memory()
    host_inputs = []
    for r in range(rounds):
        first = Wm if r == 0 else 0
        # after the timed, event and (without hybrid layers) graph passes
        lens_e = lens0[r] + first + (2 if hybrid else 3) * steps_in_round[r]
        n = steps_in_round[r] + (Wm if r == 0 else 0)
        g = make_inputs(cfg, lens_e, n, caches[r][1], dev, stream)
        host_inputs.append(tuple(None if x is None else x.cpu().pin_memory() for x in g))
        del g
        e_bytes += sum(kv_bytes_per_step(cfg, lens_e + (Wm if r == 0 else 0) + s)
                       for s in range(steps_in_round[r]))
    torch.cuda.synchronize()

    def step_host(c, hin, s):
        for layer in range(n_layers):
            if kinds[layer] in HYBRID:
                full = kinds[layer] == 2
                c.append_hybrid_host(layer, hin[0][s, layer], hin[1][s, layer], hin[2][s, layer],
                                     ones, k_global=hin[3][s, layer] if full else None,
                                     v_global=hin[4][s, layer] if full else None, out=hout,
                                     stream=stream)
            else:
                c.append_host(layer, hin[0][s, layer], hin[1][s, layer], hin[2][s, layer], ones,
                              out=hout, stream=stream)
        c.advance(ones, stream=stream)

    for s in range(Wm):
        step_host(caches[0][0], host_inputs[0], s)
    torch.cuda.synchronize()
    barrier()
    e0.record(stream)
    for r in range(rounds):
        first = Wm if r == 0 else 0
        for s in range(first, first + steps_in_round[r]):
            step_host(caches[r][0], host_inputs[r], s)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = e0.elapsed_time(e1)

    # ---- max over ranks
    if world > 1:
        (ms, ms_e2e, ms_graph), (alg_bytes, e_bytes, graph_bytes) = reduce_over_ranks(
            [ms, ms_e2e, ms_graph or 0.0], [alg_bytes, e_bytes, graph_bytes], dev)
    for c, _ in caches:
        c.close()
    if rank != 0:
        return None
    value = alg_bytes / (ms / 1e3) / 1e9
    tok_s = world * B * K / (ms / 1e3)
    dec = prof["decode"]
    achieved = dec["bytes"] / (dec["ms"] / 1e3) / 1e9 if dec["ms"] > 0 else None
    traffic = traffic_record("decode.cu", args.workload)
    roofline = {
        "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
        "frac": (achieved / peak) if achieved else None,
        "traffic": (traffic["dram_bytes_per_launch"] if traffic else None),
        "kernel": "decode_kernel (split-K GQA decode, tensor-core QK/PV, TMA-staged)",
        "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth, burst)",
        "alg_bytes_per_launch": dec["bytes"] / max(1, dec["launches"]),
        "avg_launch_ms": dec["ms"] / max(1, dec["launches"]),
        "frac_of_nominal_8TBs": (achieved / NOMINAL_HBM_GBS) if achieved else None,
        "by_layer_kind": split,
        "timing": "CUDA events around every library launch on the launch stream, over a "
                  "second pass of the same number of steps per cache (the timed region "
                  "runs without them)",
    }
    line = {
        "metric": METRICS.get(args.workload, METRIC), "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(decode_config(args, cfg, world), start=START_NOTE),
        "tokens_per_s": tok_s,
        "frac_of_nominal_8TBs": value / NOMINAL_HBM_GBS,
        "frac_of_measured_hbm": value / peak,
        "step_ms": per_step,
        "steady_value": (alg_bytes / K) / (per_step["median"] / 1e3) / 1e9 if per_step else None,
        "host_ms_per_step": host_ms / K,
        "roofline": roofline,
        "e2e": {"value": e_bytes / (ms_e2e / 1e3) / 1e9, "unit": "GB/s",
                "tokens_per_s": world * B * K / (ms_e2e / 1e3),
                "h2d_bytes_per_step": sum(B * (Hq + (4 if k == 2 else 2) * Hk) * D * 2
                                          for k in kinds),
                "d2h_bytes_per_step": n_layers * B * Hq * D * 2},
        "graph": {"value": graph_bytes / (ms_graph / 1e3) / 1e9, "unit": "GB/s",
                  "ms_per_step": ms_graph / K,
                  "api": "kv_step_graph_launch: one CUDA-graph replay per step (all layers "
                         "and the advance), inputs already on the device"} if ms_graph else None,
        "gpu_launches": launches,
        "kernels": {k: {"launches": p["launches"], "ms": p["ms"]} for k, p in prof.items()},
        "clocks": clk,
        "fill_s": t_fill,
        "prefill": {"kernel": "prefill_kernel (chunked prefill, 64-token chunks, cache fill)",
                    "launches": pre["launches"], "ms": pre["ms"],
                    "tflops": pre["flops"] / (pre["ms"] / 1e3) / 1e12 if pre["ms"] else None,
                    "frac_of_bf16_sustained": (pre["flops"] / (pre["ms"] / 1e3) / 1e12
                                               / peak_tflops()) if pre["ms"] else None,
                    "flops_counted": "4*Hq*D per visible (query, key) pair, causal only"},
    }
    if world == 1 and not args.no_cpu_baseline and not sub:
        gbs, tps, nr, thr, t = oracle_sample(cfg, lens0[0] + Wm + per_round, caches[0][1],
                                             budget_s=15.0)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": thr, "kind": "oracle",
                                "tokens_per_s": tps,
                                "sample": f"{nr} row-decodes of one step of the workload (all "
                                          f"{Hq} heads over each row's whole history), "
                                          f"{t:.1f} s of oracle time (at most 45 s of wall "
                                          f"time with the inputs' generation)"}
    return line


# ---------------------------------------------------------------- continuous batching

def cont_plan(cfg, n_steps, seed):
    """Initial lengths and n_steps steps of the continuous-batch mix: per step the rows
    reset first (5% of B) and every row's n_new; lengths stay within max_len."""
    rng = np.random.default_rng(seed)
    B = cfg["B"]
    lens0 = rng.integers(cfg["lo"], cfg["hi"] + 1, size=B).astype(np.int64)
    lens, steps = lens0.copy(), []
    for _ in range(n_steps):
        resets = rng.choice(B, size=max(1, B // 20), replace=False)
        lens[resets] = 0
        u = rng.random(B)
        n = np.where(u < 0.4, 1, np.where(u < 0.7, 0, rng.integers(2, 65, size=B)))
        n = np.minimum(n, cfg["max_len"] - lens)
        steps.append((resets.tolist(), n.astype(np.int64), lens.copy()))
        lens += n
    return lens0, steps


def cont_inputs(cfg, steps, seed, dev, stream):
    """q, k, v of every step and layer, [n_steps, n_layers, B, 64, H, D], generated on the
    device at each row's positions."""
    import torch
    import synth
    B, Hq, Hk, D, C = cfg["B"], cfg["Hq"], cfg["Hk"], cfg["D"], 64
    L = len(cfg["kinds"])
    qs = torch.empty((len(steps), L, B, C, Hq, D), dtype=torch.bfloat16, device=dev)
    ks = torch.empty((len(steps), L, B, C, Hk, D), dtype=torch.bfloat16, device=dev)
    vs = torch.empty_like(ks)
    rows = torch.arange(B, dtype=torch.int32, device=dev)
    seqs = torch.zeros(B, dtype=torch.int32, device=dev)
    for i, (_, _, lens) in enumerate(steps):
        pos0 = torch.from_numpy(lens.astype(np.int32)).to(dev)
        for layer in range(L):
            for t, x, H in ((synth.Q, qs, Hq), (synth.K, ks, Hk), (synth.V, vs, Hk)):
                synth.fill_device(x[i, layer].data_ptr(), seed, t, layer, rows.data_ptr(),
                                  seqs.data_ptr(), pos0.data_ptr(), B, C, H, D,
                                  stream.cuda_stream)
    return qs, ks, vs


def cont_oracle_sample(cfg, steps, seed, budget_s):
    """The oracle on whole rows (all layers, all of a row's new tokens) of the mix's first
    steps until about budget_s of oracle time, or three times that in wall time; returns
    (tokens/s, tokens, threads, seconds of oracle time)."""
    import oracle
    import synth
    Hq, Hk, D, W = cfg["Hq"], cfg["Hk"], cfg["D"], cfg["W"]
    spent, tokens = 0.0, 0
    wall0 = time.perf_counter()
    for _, n, lens in steps:
        for b in (int(x) for x in np.nonzero(n > 0)[0]):
            if spent >= budget_s or (tokens and time.perf_counter() - wall0 >= 3 * budget_s):
                break
            L, m = int(lens[b]), int(n[b])
            for layer, kind in enumerate(cfg["kinds"]):
                lo = max(0, L - W + 1) if kind == 1 else 0
                pos = range(lo, L + m)
                kh = synth.normal_bf16(seed, synth.K, layer, b, 0, pos, Hk, D)
                vh = synth.normal_bf16(seed, synth.V, layer, b, 0, pos, Hk, D)
                q = synth.normal_bf16(seed, synth.Q, layer, b, 0, range(L, L + m), Hq, D)
                t0 = time.perf_counter()
                oracle.attend(q, range(L, L + m), kh, vh, lo, Hq, Hk, W=W if kind == 1 else 0)
                spent += time.perf_counter() - t0
            tokens += m
        if spent >= budget_s or (tokens and time.perf_counter() - wall0 >= 3 * budget_s):
            break
    return tokens / spent, tokens, oracle.num_threads(), spent


def run_cont_batch(args, sub=False):
    """Config 5: tokens/s of the continuous-batch mix (decode rows, chunk rows, idle rows and
    resets in every step).  Three passes run the same step plan, each on a freshly filled
    cache: the timed region (no per-launch events), a pass with the library's per-launch
    events (kernel split, GB/s and TFLOP/s), and end to end through the host-buffer entry
    point."""
    import torch
    import kv_cache_incremental_gb300 as kvi
    rank, local_rank, world = dist_env()
    init_dist(local_rank, world)
    cfg = WORKLOADS[args.workload]
    B, Hq, Hk, D, C = cfg["B"], cfg["Hq"], cfg["Hk"], cfg["D"], CONT_CHUNK
    kinds = cfg["kinds"]
    K = args.steps if args.steps else cfg["steps"]
    Wm = max(3, args.warmup)
    seed = args.seed + 7919 * rank
    stream = torch.cuda.current_stream()
    dev = torch.device("cuda", local_rank)
    lens0, steps = cont_plan(cfg, Wm + K, seed)
    tokens = int(sum(int(n.sum()) for _, n, _ in steps[Wm:]))
    qs, ks, vs = cont_inputs(cfg, steps, seed, dev, stream)
    out = torch.empty((B, C, Hq, D), dtype=torch.bfloat16, device=dev)

    def fresh():
        c = kvi.KVCache(B, cfg["max_len"], Hq, Hk, D, cfg["W"], kinds, 1e4, local_rank)
        fill_cache(c, cfg, lens0, seed, stream)
        return c

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def run(c, i0, i1, host=None, after_step=None):
        for i in range(i0, i1):
            resets, n, _ = steps[i]
            c.reset(resets, stream=stream)
            nl = n.tolist()
            for layer in range(len(kinds)):
                if host is None:
                    c.append(layer, qs[i, layer], ks[i, layer], vs[i, layer], nl, out=out,
                             stream=stream)
                else:
                    c.append_host(layer, host[0][i, layer], host[1][i, layer], host[2][i, layer],
                                  nl, out=host[3], stream=stream)
            c.advance(nl, stream=stream)
            if after_step:
                after_step()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # ---- timed region (warm-up right before it, events after every step)
    c = fresh()
    clocks = ClockSampler(local_rank)
    clocks.start()
    run(c, 0, Wm)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    it = iter(evs[1:])
    hold_stream(stream)
    clocks.mark_start()
    torch.cuda.profiler.start()
    evs[0].record(stream)
    h0 = time.perf_counter()
    run(c, Wm, Wm + K, after_step=lambda: next(it).record(stream))
    host_ms = (time.perf_counter() - h0) * 1e3   # enqueue time of the K steps
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    clocks.mark_stop()
    barrier()
    clk = clocks.stop()
    ms = evs[0].elapsed_time(evs[-1])
    per_step = step_times(evs)
    c.close()
    # ---- the same steps with per-launch events
    c = fresh()
    run(c, 0, Wm)
    torch.cuda.synchronize()
    c.profile(True)
    run(c, Wm, Wm + K)
    torch.cuda.synchronize()
    prof = {k: c.profile_read(k, reset=True) for k in ("append", "decode", "prefill", "combine",
                                                     "commit", "state")}
    c.profile(False)
    c.close()
    # ---- end to end: host buffers (pinned), copies inside the timed region
    host = tuple(x.cpu().pin_memory() for x in (qs, ks, vs))
    host = host + (torch.empty((B, C, Hq, D), dtype=torch.bfloat16).pin_memory(),)
    c = fresh()
    run(c, 0, Wm, host)
    torch.cuda.synchronize()
    barrier()
    e0.record(stream)
    run(c, Wm, Wm + K, host)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = e0.elapsed_time(e1)
    c.close()
    if world > 1:
        (ms, ms_e2e), (tokens_all,) = reduce_over_ranks([ms, ms_e2e], [float(tokens)], dev)
    else:
        tokens_all = float(tokens)
    if rank != 0:
        return None
    tot_bytes = sum(p["bytes"] for p in prof.values())
    tot_flops = sum(p["flops"] for p in prof.values())
    dec, pre = prof["decode"], prof["prefill"]
    if pre["ms"] >= dec["ms"]:
        tf = pre["flops"] / (pre["ms"] / 1e3) / 1e12 if pre["ms"] else None
        roofline = {"bound": "tensor", "achieved": tf, "peak": peak_tflops(), "unit": "TFLOP/s",
                    "frac": tf / peak_tflops() if tf else None, "traffic": None,
                    "kernel": "prefill (chunk rows: tcgen05 prefill_tc_kernel and mma.sync "
                              "prefill_kernel)",
                    "peak_source": "measured bf16_tflops_sustained (kernel inside a long step)"}
    else:
        peak, kind = measured_peaks()
        gb = dec["bytes"] / (dec["ms"] / 1e3) / 1e9 if dec["ms"] else None
        roofline = {"bound": "hbm", "achieved": gb, "peak": peak, "unit": "GB/s",
                    "frac": gb / peak if gb else None, "traffic": None,
                    "kernel": "decode_kernel (decode rows)",
                    "peak_source": f"{kind} hbm_gbs (copy bandwidth, burst)"}
    roofline["timing"] = ("CUDA events around every library launch on the launch stream, over a "
                          "second pass of the same steps on a freshly filled cache")
    h2d = len(kinds) * B * C * (Hq + 2 * Hk) * D * 2
    line = {
        "metric": METRICS[args.workload],
        "value": tokens_all / (ms / 1e3), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(cont_config(args, cfg, world), start=START_NOTE),
        "gbs": tot_bytes / (ms / 1e3) / 1e9, "tflops": tot_flops / (ms / 1e3) / 1e12,
        "roofline": roofline,
        "e2e": {"value": tokens_all / (ms_e2e / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": len(kinds) * B * C * Hq * D * 2},
        "gpu_launches": sum(p["launches"] for p in prof.values()),
        "kernels": {k: {"launches": p["launches"], "ms": p["ms"],
                        "gbs": p["bytes"] / (p["ms"] / 1e3) / 1e9 if p["ms"] else None,
                        "tflops": p["flops"] / (p["ms"] / 1e3) / 1e12 if p["ms"] else None}
                    for k, p in prof.items()},
        "step_ms": per_step,
        "host_ms_per_step": host_ms / K,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline and not sub:
        tps, nt, thr, t = cont_oracle_sample(cfg, steps[Wm:], seed, budget_s=15.0)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                                "sample": f"{nt} tokens (whole rows of the first timed steps, "
                                          f"all {len(kinds)} layers), {t:.1f} s of oracle time"}
    return line


def run_reference_cont(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    cfg = WORKLOADS[args.workload]
    config = cont_config(args, cfg, world)
    if not args.steps:
        args.steps = 10
    Wm = max(3, args.warmup)
    _, steps = cont_plan(cfg, Wm + args.steps, args.seed)
    cont_oracle_sample(cfg, steps[:1], args.seed, budget_s=0.5)
    total_tok, total_t, thr = 0, 0.0, 1
    for i in range(Wm, Wm + args.steps):   # the steps the timed arm times
        _, tok, thr, t = cont_oracle_sample(cfg, steps[i:i + 1], args.seed, budget_s=1.0)
        total_tok += tok
        total_t += t
    value = total_tok / total_t
    print(json.dumps({
        "impl": "reference", "metric": METRICS[args.workload], "value": value,
        "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                         "sample": f"{total_tok} tokens (whole rows, all layers) over "
                                   f"{args.steps} steps, about 1 s of oracle time each"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


# Workloads whose records the default (headline) line carries beside its own: the
# long-context mixed layout (config 4, the >= 70% of HBM peak target) and the
# continuous-batch mix (config 5).
SUB_WORKLOADS = ("long_ctx", "cont_batch")
SUB_KEYS = ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "step_ms",
            "host_ms_per_step",
            "steady_value", "tokens_per_s", "frac_of_measured_hbm", "frac_of_nominal_8TBs",
            "gbs", "tflops", "roofline", "graph", "e2e", "gpu_launches", "kernels", "clocks",
            "config", "prefill")


def run_workload(args, sub=False):
    mix = WORKLOADS[args.workload].get("mix", False)
    return run_cont_batch(args, sub) if mix else run_ours(args, sub)


def main():
    args = parse()
    mix = WORKLOADS[args.workload].get("mix", False)
    if args.impl == "reference":
        run_reference_cont(args) if mix else run_reference(args)
        return
    if args.fill_only:
        run_fill_only(args)
        return
    line = run_workload(args)
    if args.workload == "decode_bw" and not args.no_sub_workloads and not args.max_len \
            and not args.fill_to:
        subs = {}
        for w in SUB_WORKLOADS:
            a2 = argparse.Namespace(**vars(args))
            a2.workload = w
            rec = run_workload(a2, sub=True)
            if rec is not None:
                subs[w] = {k: rec[k] for k in SUB_KEYS if k in rec}
        if line is not None:
            line["workloads"] = subs
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
