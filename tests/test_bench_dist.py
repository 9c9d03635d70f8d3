"""bench.py's multi-process path on CPU (gloo, world size 2).

The method has no exchange step, so N GPUs run N independent replicas; the
only cross-rank operations are the barrier and the max-over-ranks time that
turns per-rank timings into the whole-job rate.  Those run here on two gloo
ranks, plus the rules of the reference arm under torchrun (rank 0 alone
prints) and the warm-up floor.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out_dir: str):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                       # rank 1 is the slower one
        worst = bench.max_over_ranks(ms, world)
        rate = bench.whole_job_rate(1e12, 4, world, worst)
        dist.barrier()
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"worst": worst, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_on_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    got = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for g in got:
        assert g["worst"] == 15.0                     # both ranks see the slowest rank's time
        # 2 replicas x 4 steps x 1e12 flop in 15 ms
        assert abs(g["rate"] - 2 * 4 * 1e12 / 15e-3 / 1e12) < 1e-9


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert abs(bench.whole_job_rate(2e12, 10, 1, 1000.0) - 20.0) < 1e-12


def test_reference_arm_non_zero_rank_prints_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_warmup_floor_is_enforced():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "warmup" in r.stderr


@pytest.mark.parametrize("steps", [1])
def test_reference_arm_prints_one_line(steps):
    # the reference arm is the CPU oracle: runs here, on a small bounded sample
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", str(steps),
                        "--warmup", "3", "--workload", "relu_1024"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
