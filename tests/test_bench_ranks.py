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


def test_algorithmic_bytes_follow_the_pages_accounting():
    # 132 B of index-K per context token, read once per request and full layer,
    # plus 656 B per selected latent row (at most 2048 per query row) per layer;
    # the 1M-token decode batch and the tiny case by hand, the 32K batch by sum
    import bench
    import synth
    w = synth.workload("decode1m")
    idx, kv = bench.workload_bytes(w)[:2]
    assert idx == 4 * 1_048_576 * 132 and kv == 4 * 2048 * 656
    assert idx + kv == 559_022_080
    w = synth.workload("decode32k")
    idx, kv = bench.workload_bytes(w)[:2]
    assert w.layers == ["full", "shared", "shared", "shared"]
    assert idx == 132 * sum(w.seq_len)
    assert kv == 4 * 656 * sum(min(2048, L) for L in w.seq_len)
    t = synth.workload("tiny")
    idx, kv = bench.workload_bytes(t)[:2]
    assert idx == 132 * t.seq_len[0] and kv == 656 * min(2048, t.seq_len[0]) * len(t.layers)
    # an MXFP4 index cache: 68 B per token instead of 132
    m = synth.workload("decode1m")
    m.index_format = "mxfp4"
    assert bench.workload_bytes(m)[0] == 4 * 1_048_576 * 68


def test_launch_count_follows_the_sparse_mla_split():
    # 152 SMs: 1..19 decode rows take one CTA per tile (partials, combine kernel);
    # 20..38 rows run as clusters of 4 and 39..76 as clusters of 2 (merged in
    # the cluster); 77..152 rows one CTA each (written whole); 153..1215 rows
    # equal shares (combine kernel); 1216 and more whole rows per CTA
    import bench
    k = bench.kernels_per_call
    for rows, n in [(1, 2), (4, 2), (19, 2), (20, 1), (38, 1), (39, 1), (64, 1), (76, 1), (77, 1), (100, 1),
                    (152, 1), (153, 2), (1215, 2), (1216, 1), (8192, 1)]:
        assert k("sparse_mla_decode", rows, 152) == n, rows
    assert k("indexer_topk", 64, 152) == 4 and k("index_k_store", 64, 152) == 1
