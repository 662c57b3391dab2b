"""Multi-rank host logic of the benchmark (one replica per rank, weak scaling) on gloo
ranks on the CPU: rank environment, max-over-ranks timing, whole-job rate, launch
totals, per-rank seeds, and the reference arm running on rank 0 only."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import multirank_worker

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [2])
def test_gloo_ranks_reduce_and_rate(tmp_path, world):
    mp.spawn(multirank_worker.rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    recs = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, rec in enumerate(recs):
        assert rec["env"] == [r, world, r]
        assert rec["max"] == 3 * (world - 1) + 1
        assert rec["job"] == [2.0, world * 10 / 2.0]  # slowest rank's time, every rank's steps
        assert rec["sum"] == sum(x + 3 for x in range(world))
    # every rank draws its own replica of the workload
    assert len({rec["seed"] for rec in recs}) == world
    assert len({rec["q_sum"] for rec in recs}) == world


def test_single_rank_helpers_need_no_process_group():
    import bench

    assert bench.reduce_max(1.5, 1) == 1.5
    assert bench.job_rate(20, 0.5, 1) == (0.5, 40.0)
    assert bench.sum_over_ranks(7, 1) == 7
    bench.barrier(1)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
