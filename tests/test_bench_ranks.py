"""bench.py's multi-rank logic on CPU: gloo, world size 2.

Every rank runs the full per-GPU workload (weak scaling, no data exchange); the
job's time is the slowest rank's and its rate counts the work of all ranks.
"""

import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(1.5 + rank, dist, "cpu")  # rank 1 is the slow one
    out[rank] = (t, bench.whole_job_rate(10.0, world, 4, t))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_rate_gloo():
    world = 2
    port = 29500 + (os.getpid() % 1000)
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        t, rate = res[rank]
        assert t == 2.5
        assert rate == pytest.approx(world * 10.0 * 4 / 2.5)


def test_single_process_helpers():
    import bench

    assert bench.max_over_ranks(3.0, None) == 3.0
    assert bench.whole_job_rate(2.0, 1, 5, 2.0) == 5.0


def test_reference_arm_only_rank0_prints():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
