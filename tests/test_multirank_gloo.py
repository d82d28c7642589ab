"""Multi-rank paths on CPU ranks over gloo: the benchmark's (one process per
rank at world size 2, the slowest rank's time taken as the job's, the
reference arm on rank 0 only) and the sharded PatchGroupNorm exchange (one
all-gather of per-patch partials at world size 3)."""
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


def _gn_rank(rank, world, port, q):
    # The sharded PatchGroupNorm exchange on CPU ranks: every rank holds one
    # patch of the activation, computes its (count, mean, M2) per (sample,
    # group), and one all-gather of those partials gives every rank the pooled
    # mean and biased variance of the whole tensor (the pages need two
    # all-reduces for it).
    sys.path.insert(0, ROOT)
    import numpy as np
    from oracle import groupnorm as GN
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(3)
        x = rng.standard_normal((2, 12, 10, 14)) * 1.5
        sizes = [4, 3, 3][:world]                     # ragged height bands
        starts = np.cumsum([0] + sizes[:-1])
        patches = [x[:, :, s:s + n] + (r - 1) * 2.0 for r, (s, n) in enumerate(zip(starts, sizes))]
        cnt, mean, m2 = GN.patch_partials([patches[rank]], 4)
        mine = torch.from_numpy(np.stack([cnt[0].astype(np.float64), mean[0], m2[0]], axis=-1))
        got = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(got, mine)
        c = np.stack([g[..., 0].numpy() for g in got])
        m = np.stack([g[..., 1].numpy() for g in got])
        v = np.stack([g[..., 2].numpy() for g in got])
        n = c.sum(0)
        mu = (c * m).sum(0) / n
        var = (v + c * (m - mu) ** 2).sum(0) / n
        ref_mu, ref_var = GN.group_stats(patches, 4)
        ok = np.abs(mu - ref_mu).max() < 1e-12 and np.abs(var / ref_var - 1).max() < 1e-12
        q.put((rank, bool(ok)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_groupnorm_partials_all_gather_gives_the_pooled_statistics():
    world = 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gn_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert sorted(q.get(timeout=10) for _ in range(world)) == [(r, True) for r in range(world)]
