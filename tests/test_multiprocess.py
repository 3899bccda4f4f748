"""The multi-process path of bench.py on CPU: world size 2 over gloo.

Sequences are independent, so N GPUs run N replicas with no collective on the data path;
the only cross-rank steps are the timing reduction (max over ranks) and rank 0 printing
the line.  Both are exercised here without a GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                     # rank 1 is the slow one
        out[rank] = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn")
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_max_over_ranks_without_process_group():
    assert bench.max_over_ranks(3.5, None, torch.device("cpu")) == 3.5


def test_whole_job_rate_adds_the_replicas():
    # 2 ranks x 100 steps in at most 50 ms -> 4000 steps/s for the job
    assert bench.whole_job_rate(2, 100, 50.0) == pytest.approx(4000.0)
    assert bench.whole_job_rate(1, 100, 50.0) == pytest.approx(2000.0)


def test_reference_arm_under_torchrun_prints_one_line():
    """`bench.py --impl reference` launched with two ranks: rank 0 times the oracle on the
    tiny workload and prints one JSON line; rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--steps", "2", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["unit"] == "steps/s" and rec["value"] > 0
    assert rec["config"]["workload"] == "tiny"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
