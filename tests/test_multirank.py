"""The N > 1 path of bench.py on CPU: two gloo ranks, each timing its own replica.

The job's time is the slowest rank's (max over ranks) and the job's value is
the flops of all replicas over that time.  No GPU is involved.
"""
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, per_rank_ms, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.reduce_max(dist, per_rank_ms[rank], "cpu")
        value = bench.job_tflops(2.0 * 1024 ** 3, ms, world)
        out[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_max_and_sum_the_replicas():
    world = 2
    per_rank_ms = [1.25, 2.5]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), per_rank_ms, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, value = res[rank]
        assert ms == 2.5                                     # the slowest rank's time
        assert value == pytest.approx(world * 2.0 * 1024 ** 3 / 2.5e-3 / 1e12)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(None, 3.5, "cpu") == 3.5
    assert bench.job_tflops(1e12, 1000.0, 1) == pytest.approx(1.0)


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
