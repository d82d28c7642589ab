"""The benchmark's multi-GPU path on CPU ranks: one process per rank over
gloo at world size 2, the slowest rank's time taken as the job's, and the
reference arm running on rank 0 only."""
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
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank           # rank 1 is the slowest
        slow = bench.max_over_ranks(torch, dist, world, ms, torch.device("cpu"))
        rate = bench.whole_job_gbs(1e9, slow, world)
        out.put((rank, slow, rate))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time_and_rates_add_up():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slow, rate in got:
        assert slow == 15.0
        assert abs(rate - 2 * 1e9 / 15e-3 / 1e9) < 1e-9


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
