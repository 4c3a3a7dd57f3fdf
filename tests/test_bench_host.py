"""Host-side logic of bench.py that needs no GPU: the continuous-batch step plan, the
algorithmic byte count of a decode step, and the reference arm's JSON lines."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_cont_plan_follows_the_mix():
    cfg = bench.WORKLOADS["cont_batch"]
    B = cfg["B"]
    lens0, steps = bench.cont_plan(cfg, 300, seed=3)
    assert lens0.min() >= cfg["lo"] and lens0.max() <= cfg["hi"]
    lens = lens0.copy()
    counts = np.zeros(3)
    for resets, n, before in steps:
        assert len(resets) == max(1, B // 20) == len(set(resets))
        lens[resets] = 0
        assert np.array_equal(before, lens)        # positions the step starts from
        assert (n >= 0).all() and (n <= 64).all() and (lens + n <= cfg["max_len"]).all()
        counts += [(n == 1).sum(), (n == 0).sum(), (n >= 2).sum()]
        lens += n
    frac = counts / counts.sum()
    assert abs(frac[0] - 0.4) < 0.02 and abs(frac[1] - 0.3) < 0.02 and abs(frac[2] - 0.3) < 0.02
    again = bench.cont_plan(cfg, 300, seed=3)
    assert np.array_equal(again[0], lens0)
    assert all(np.array_equal(a[1], b[1]) for a, b in zip(again[1], steps))


def test_step_bytes_by_layer_kind():
    """Every visible K/V byte once per kv head, plus the new keys' and the queries' traffic:
    a hybrid layer reads its group's keys 0..p and its window; a full hybrid layer also takes
    the group's new global key."""
    base = dict(B=2, Hq=8, Hk=2, D=64, max_len=4096, W=16, lo=0)
    lens = np.array([10, 100])
    B, Hq, Hk, D, W = 2, 8, 2, 64, 16

    def new_bytes(streams):
        return B * (Hq + 2 * streams * Hk) * D * 2 + 2 * streams * B * Hk * D * 2 + B * Hq * D * 2

    def kv(keys):
        return float(np.sum(2.0 * Hk * keys * D * 2))

    local = np.minimum(lens + 1, W)
    expect = {0: kv(lens + 1) + new_bytes(1), 1: kv(local) + new_bytes(1),
              2: kv(lens + 1 + local) + new_bytes(2), 3: kv(lens + 1 + local) + new_bytes(1)}
    for kind, want in expect.items():
        got = bench.kv_bytes_per_step(dict(base, kinds=[kind]), lens)
        assert got == want, kind
    both = bench.kv_bytes_per_step(dict(base, kinds=[2, 3, 1]), lens)
    assert both == expect[2] + expect[3] + expect[1]


def _reference_line(workload):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", workload, "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_reference_arm_lines_carry_the_timed_arms_config():
    """The reference arm reports the timed arm's metric unit and its exact config (the same
    function builds both), with the oracle as its CPU baseline."""
    for workload, unit in (("cont_batch", "tokens/s"), ("decode_bw", "GB/s")):
        d = _reference_line(workload)
        assert d["impl"] == "reference" and d["unit"] == unit and d["value"] > 0
        args = bench.parse(["--workload", workload, "--steps", "1", "--warmup", "1"])
        cfg = bench.WORKLOADS[workload]
        want = (bench.cont_config if cfg.get("mix") else bench.decode_config)(args, cfg, 1)
        assert d["config"] == want and d["metric"] == bench.METRICS[workload]
        assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
        assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
