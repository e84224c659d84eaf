"""The multi-GPU path of bench.py on the CPU: world_size 2, gloo backend.

bench.py runs N independent replicas (one per GPU, no collective on the data
path); only the whole-job aggregation talks across ranks: the tokens of all
ranks over the slowest rank's timed region.
"""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r processed 16*(r+1) tokens in (r+1)*0.5 s
    v, tmax = bench.job_throughput(16 * (rank + 1), 0.5 * (rank + 1), True, "cpu")
    q.put((rank, v, tmax))
    dist.barrier()
    dist.destroy_process_group()


def test_job_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for _, v, tmax in got:
        assert tmax == pytest.approx(1.0)
        assert v == pytest.approx((16 + 32) / 1.0)


def test_single_rank_throughput():
    sys.path.insert(0, ROOT)
    import bench
    v, t = bench.job_throughput(32, 0.25, False, "cpu")
    assert v == 128 and t == 0.25


def test_reference_arm_non_zero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
