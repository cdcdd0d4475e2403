"""The N>1 host logic of bench.py on CPU ranks (gloo, world size 2): each rank
draws its own batch, the slowest rank's time is taken, and the whole-job
throughput counts every rank's units.  The attention path itself has no
collective (sequences are independent)."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [1.5 + rank, 10.0 - rank]          # rank 1 is slower on the first, faster on the second
    got = bench.max_over_ranks(ms, world, "cpu")
    seed = bench.rank_seed(1001, rank)
    seeds = [None] * world
    dist.all_gather_object(seeds, seed)
    q.put((rank, got, seeds))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_distinct_batches():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, seeds in res:
        assert got == [2.5, 10.0]
        assert len(set(seeds)) == world


def test_job_throughput_counts_all_ranks():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(64, 1, 1.0) == pytest.approx(64000.0)
    assert bench.job_throughput(64, 4, 2.0) == pytest.approx(128000.0)
    assert bench.max_over_ranks([3.0, 4.0], 1, "cpu") == [3.0, 4.0]


def test_reference_arm_only_rank0_prints():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
