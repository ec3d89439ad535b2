"""bench.py's multi-rank logic on the CPU: two gloo ranks on 127.0.0.1 (no GPU).

Each rank runs the whole workload as a replica; the job's step time is the
slowest rank's and the job's rate counts the units of every rank.  The
reference arm runs on rank 0 only; the other ranks exit without work.
"""
import io
import os
import pathlib
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = pathlib.Path(__file__).resolve().parent.parent
sys.path.insert(0, str(ROOT))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step = bench.slowest_rank(1.0 + rank, world)          # rank r took 1 + r ms
        out[rank] = (step, bench.job_rate(1e6, world, step))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    for rank in range(world):
        step, rate = res[rank]
        assert step == 2.0                                      # the slower rank's 2 ms
        assert rate == pytest.approx(1e6 * world / 2e-3)       # both ranks' units over that time


def test_single_rank_passes_through():
    import bench
    assert bench.slowest_rank(3.5, 1) == 3.5
    assert bench.job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.main.__globals__["argparse"].Namespace(workload="tiny", steps=1, warmup=0, cpu_seconds=0.5)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    assert buf.getvalue() == ""


def test_reference_arm_prints_one_json_line():
    import json
    import subprocess
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "1", "--cpu-seconds", "1"],
                       capture_output=True, text=True, timeout=300, cwd=str(ROOT),
                       env={**os.environ, "RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["cores"] == 1 and d["cpu_baseline"]["threads"] == 1 and d["cpu_baseline"]["cpu_model"]


def test_cpu_baseline_leg_runs_the_oracle_on_one_core():
    # the GPU arm's cpu_baseline leg: a child process with every BLAS / OpenMP pool at one thread,
    # pinned to one core, timing the oracle on the first scoring layer of the same workload
    import bench
    args = bench.main.__globals__["argparse"].Namespace(workload="tiny", chunk=0, budget=0)
    d = bench.cpu_baseline(args, budget_s=0.5)
    assert d["kind"] == "oracle" and d["value"] > 0 and d["cores"] == 1 and d["threads"] == 1
    assert "scoring layer 0" in d["sample"]
