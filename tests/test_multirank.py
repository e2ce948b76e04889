"""The multi-GPU bench path is independent replicas: each rank runs its own
workload and the only cross-rank step is the timing reduction.  Two gloo
ranks on CPU exercise that reduction and the whole-job throughput arithmetic."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        slow = bench.max_over_ranks(10.0 + 5.0 * rank)          # rank 1 is the slow one
        seed = bench.replica_seed(20260002, rank)
        value = bench.job_throughput(1e9, 100, world, slow)
        results[rank] = (slow, seed, value)
    finally:
        dist.destroy_process_group()


def test_replica_timing_uses_the_slowest_rank_and_sums_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.start_processes(_worker, args=(world, port, results), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(results)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] != res[1][1]
    # 2 ranks x 100 steps x 1 GB over the slowest rank's 15 ms
    assert res[0][2] == pytest.approx(2 * 100 * 1e9 / 0.015 / 1e9)


def test_single_process_reduction_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(2e9, 10, 1, 20.0) == pytest.approx(1000.0)


def test_bench_gpus_2_launches_two_ranks_itself():
    """`bench.py --gpus 2` run without a launcher starts two ranks itself
    (torch.distributed.run on 127.0.0.1); the dry run swaps the GPU work for
    a host loop, so the launch, the gloo barrier and the reductions run here
    without a GPU.  Both ranks report, and n_gpus is the ranks that ran."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--dry-run",
                        "--steps", "3", "--warmup", "1"], capture_output=True, text=True, timeout=240,
                       env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["dry_run"] and line["n_gpus"] == 2 and line["ranks_reported"] == 2
    assert len(line["rank_ms"]) == 2 and line["slowest_ms"] == max(line["rank_ms"])
