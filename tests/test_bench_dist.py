"""The replicas path of bench.py with two gloo ranks on CPU (no GPU, no NCCL)."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    times, units = bench.reduce_over_ranks([1.0 + rank, 10.0 * (rank + 1)],
                                           [100.0 * (rank + 1), 7.0], "cpu")
    assert bench.dist_env() == (rank, rank, world)
    dist.destroy_process_group()
    q.put((rank, times, units))


def test_two_gloo_ranks_take_max_time_and_sum_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, times, units in res:
        assert times == [2.0, 20.0]
        assert units == [300.0, 14.0]


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    small = dict(B=2, Hq=4, Hk=2, D=64, max_len=300, W=0, kinds=[0], lo=100, steps=2,
                 per_round=2)
    monkeypatch.setitem(bench.WORKLOADS, "tiny", small)
    args = bench.parse(["--workload", "tiny", "--steps", "2", "--warmup", "1"])
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    assert buf.getvalue() == ""
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["n_gpus"] == 2
    assert line["config"] == bench.decode_config(args, small, 2)
    assert line["e2e"]["h2d_bytes_per_step"] == 0
