"""The multi-process (replicas, one rank per GPU) path of bench.py, on CPU.

bench.py --gpus N runs N independent replicas of the step, one per rank,
times each with CUDA events and reports the whole job: every rank's tokens
over the slowest rank's time.  The cross-rank pieces are checked here with
two gloo ranks, and the reference arm under torchrun (rank 0 alone runs and
prints; the other ranks exit 0 without work).
"""
import argparse
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.5 + rank, dist)       # rank 1 is the slower one
        q.put((rank, ms, bench.job_value(755, world, ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_times_the_job_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in got:
        assert ms == 2.5                                   # the max over ranks, on every rank
        assert value == pytest.approx(755 * 2 / 2.5e-3)    # both ranks' tokens over the slowest time


def test_one_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_value(100, 1, 2.0) == pytest.approx(50_000.0)


def test_reference_arm_on_a_nonzero_rank_does_no_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(impl="reference", gpus=2, steps=1, warmup=0, workload=1)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_under_torchrun_two_ranks():
    """torchrun with two ranks on 127.0.0.1: exactly one JSON line (rank 0)."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "2", "--warmup", "0", "--workload", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["config"]["workload"] == "layout-example-N9"


def test_gpus_two_without_torchrun_relaunches_as_two_ranks():
    """bench.py --gpus 2 started as one plain process re-runs itself under
    torch.distributed.run with two ranks: one JSON line, n_gpus 2."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "0",
           "--workload", "1"]
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    env["OMP_NUM_THREADS"] = "1"
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


def test_gpus_flag_must_match_the_launched_ranks():
    """A WORLD_SIZE that disagrees with --gpus is refused before any work."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "1"]
    env = dict(os.environ, WORLD_SIZE="3", RANK="0", OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=120, env=env)
    assert res.returncode == 2
    assert "WORLD_SIZE=3" in res.stderr and not res.stdout.strip()


def test_reference_arm_line_carries_the_contract_keys():
    """One process: the reference arm's JSON line has every key of the
    benchmark contract, its e2e moves no bytes, and its value is tokens over
    the measured step time."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "0", "--workload", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] >= 3
    assert d["higher_is_better"] is True and d["unit"] == "query tokens/s"
    assert d["value"] == pytest.approx(9 / (d["ms_per_step"] * 1e-3))           # 9 query tokens per step
    assert d["config"]["workload"] == "layout-example-N9"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
