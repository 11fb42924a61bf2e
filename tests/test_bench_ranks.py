"""Multi-rank logic of bench.py on CPU ranks (gloo, world size 2).

The step runs one replica per rank with no exchange on the data path; the
only collective is the maximum of the timings, and rank 0 alone prints.
"""
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [1.0 + rank, 10.0 - rank]             # rank 1 slower in the first, faster in the second
    got = bench.max_over_ranks(mine, "cpu")
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    world = 2
    port = 29500 + os.getpid() % 1000
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert out[0] == [2.0, 10.0] and out[1] == [2.0, 10.0]


def test_job_throughput_is_weak_scaling():
    import bench
    one = bench.job_throughput(64, 1, 0.5)
    assert one == pytest.approx(128000.0)
    assert bench.job_throughput(64, 4, 0.5) == pytest.approx(4 * one)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
