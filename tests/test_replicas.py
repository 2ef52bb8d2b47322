"""The multi-rank host logic of bench.py, on CPU ranks over gloo (world size 2).

The path shards into independent replicas: every rank decodes its own batch
(seeded apart), nothing is exchanged on the data path, the timed region is
the slowest rank's, and only rank 0 runs the reference arm and prints.
"""
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_minmax_gb300 import workloads

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(10.0 + rank, dist, "cpu")
        cfg = workloads.scaled(workloads.CONFIGS[1], S=256, K=4)
        wl = workloads.generate(cfg, device="cpu", seed=bench.replica_seed(cfg, rank))
        q.put((rank, slowest, bench.replica_seed(cfg, rank), float(wl.q.float().sum()), float(wl.k_pool.float().sum())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_decode_distinct_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [11.0, 11.0]  # both ranks report the slowest rank's time
    assert res[0][2] != res[1][2]  # seeded apart
    assert (res[0][3], res[0][4]) != (res[1][3], res[1][4])  # distinct replicas of the workload


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == ""


def test_max_over_ranks_alone_is_the_value():
    import bench

    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25
