"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The layer does not shard: N GPUs run N independent replicas, and the only
cross-rank steps are the barriers around the timed region and the maximum of
the ranks' times.  These tests run that logic as two gloo ranks on the CPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.rank_env() == (world, rank, rank)
        bench.barrier()
        # rank r "took" 1.5 + 3 r seconds: every rank must see the slowest
        slowest = bench.max_over_ranks(1.5 + 3.0 * rank)
        rate = bench.whole_job_rate(512 * 10, world, slowest)
        bench.barrier()
        with open(os.path.join(outdir, "r%d.json" % rank), "w") as f:
            json.dump({"slowest": slowest, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / ("r%d.json" % r))) for r in range(world)]
    for r in res:
        assert r["slowest"] == 4.5
        # 512 tokens x 10 steps on each of 2 replicas over the slowest 4.5 s
        assert r["rate"] == pytest.approx(2 * 5120 / 4.5)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.25) == 2.25
    bench.barrier()
    assert bench.whole_job_rate(100, 1, 0.5) == 200


def test_reference_arm_runs_on_rank_zero_only():
    # a non-zero rank of the reference arm exits 0 without work or output
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
