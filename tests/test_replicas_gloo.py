"""The multi-rank bench path on CPU: world size 2 over gloo.

The attention shards into independent replicas (one per GPU, no collective on
the data path); the only cross-rank steps are the barrier around the timed
region and the max-over-ranks reduction of the elapsed time, from which the
whole-job throughput is formed.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank)    # rank 1 is the slow one
        value = bench.job_throughput(world, 4, 10 ** 12, slowest)
        out[rank] = (slowest, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replica_ranks_agree_on_the_slowest_time():
    world = 2
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slowest, value = res[0]
    assert slowest == 15.0
    # 2 ranks x 4 steps x 1 TFLOP in 15 ms.
    assert value == pytest.approx(2 * 4 * 1.0 / 15e-3)


def test_single_process_reduction_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(1, 10, 2 * 10 ** 12, 1000.0) == pytest.approx(20.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm (the oracle on the host cores) runs on
    rank 0 alone: another rank exits 0 at once and prints nothing."""
    import subprocess
    import sys
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"],
                         env=env, capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == ""
