"""The N > 1 path of bench.py on CPU: gloo ranks at world size 2.

bench.py runs one independent replica of the decode step per GPU (the path has
no exchange step), takes each timing's maximum over ranks and reports the
whole-job time per step.  These tests run that aggregation with two gloo
processes, and check that the oracle arm leaves ranks other than 0 idle.
"""

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


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r saw a step time of 10 + r and an end-to-end time of 50 - r
        got = bench.max_over_ranks([10.0 + rank, 50.0 - rank])
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(got, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        with open(tmp_path / f"rank{r}.json") as f:
            assert json.load(f) == [11.0, 50.0]  # every rank holds the maxima


def test_max_over_ranks_without_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks([3.5, 7]) == [3.5, 7.0]


def test_whole_job_time_counts_all_replicas():
    # two replicas each finishing a step in 20 us complete two steps per 20 us
    assert bench.whole_job_us(20.0, 2) == pytest.approx(10.0)
    assert bench.whole_job_us(13.0, 1) == pytest.approx(13.0)


def test_reference_arm_only_on_rank_0():
    assert bench.runs_reference_arm(0)
    assert not bench.runs_reference_arm(1)
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3",
                        "--workload", "tiny_b1_h16_e4m3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
