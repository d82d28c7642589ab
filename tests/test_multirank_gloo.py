"""Multi-rank paths on CPU ranks over gloo: the benchmark's (one process per
rank at world size 2, the slowest rank's time taken as the job's, the
reference arm on rank 0 only), the row- and frame-sharded stitch (the
library's rank layout and patch_groupnorm_gb300.sharded's own entry points
at world sizes 2 and 3, the CPU oracle standing in for the kernels on every
rank),
and the sharded PatchGroupNorm (every rank's records in the library's layout,
one all-gather, pooled to the unsharded statistics)."""
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


def _spawn(target, world, *args):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q) + args) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return dict(got)


# --------------------------------------------------------------------------
# row-sharded stitch: the library's rank layout, the module's halo exchange
# over gloo, the oracle standing in for the stitch kernel on each rank's grid
# --------------------------------------------------------------------------

STITCH_CASES = {
    # name: (frame axis or None, height axis, width axis, B, C)
    "image": (None, (56, 16, 0.25, 8), (40, 16, 0.25, 8), 2, 3),
    "sliver": (None, (50, 16, 0.25, 4), (24, 8, 0.5, 4), 1, 2),
    "video": ((21, 8, 0.25, 1), (40, 16, 0.25, 4), (24, 16, 0.25, 4), 1, 2),
}


def _stitch_tiles(case):
    import numpy as np
    from oracle.geometry import axis_layout
    at, ay, ax, B, C = STITCH_CASES[case]
    lt = axis_layout(*at) if at else None
    ly, lx = axis_layout(*ay), axis_layout(*ax)
    rng = np.random.default_rng(len(case))
    frames = lt.extents if lt else [None]
    tiles = [[[torch.from_numpy(rng.uniform(-1, 1, (B, C) + ((f,) if f else ()) + (h, w))).to(torch.bfloat16)
               .view(torch.int16) for w in lx.extents] for h in ly.extents] for f in frames]
    return lt, ly, lx, B, C, tiles


def _local_axis(ly, row_begin, row_end, halo_rows):
    # the rank's grid rows, preceded by the received band as a tile of
    # halo_rows rows (blend and crop rules unchanged)
    from oracle.geometry import AxisLayout
    ext = ([halo_rows] if halo_rows else []) + ly.extents[row_begin:row_end]
    blends = [0] + [min(ext[n - 1], ext[n], ly.blend_extent) for n in range(1, len(ext))]
    kept = [min(L, ly.row_limit) for L in ext]
    offs = [sum(kept[:n]) for n in range(len(kept))]
    return AxisLayout(ly.stride, list(range(len(ext))), ext, ly.blend_extent, ly.row_limit, blends, kept, offs,
                      sum(kept))


class _OracleLib:
    """The calls of the library binding that patch_groupnorm_gb300.sharded
    makes, on CPU tensors, for CPU ranks: the rank layout from the library's
    host-only call, the stitch of a rank's grid (the received band as its
    first tile row) and the GroupNorm records and pooling from the CPU
    oracle and plain float64 arithmetic.  Test infrastructure only."""

    def __init__(self, tb):
        self.tb = tb

    def tb_stitch_shard_layout(self, *args):
        return self.tb.tb_stitch_shard_layout(*args)

    @staticmethod
    def _lay(a):
        from oracle.geometry import axis_layout
        return axis_layout(a.latent_extent, a.latent_tile, a.overlap, a.scale)

    def tb_stitch_halo_pack(self, row_tiles, at, ay, ax, row, halo):
        e = self._lay(ay).blends[row + 1]
        flat = list(row_tiles) if at is None else [t for per_k in row_tiles for t in per_k]
        halo.copy_(torch.cat([t[..., -e:, :].reshape(-1) for t in flat]))

    def _shard(self, tiles3, halo, at, ay, ax, rb, re_, out):
        import numpy as np
        from oracle.stitch import stitch as oracle_stitch
        lt = self._lay(at) if at is not None else None
        ly, lx = self._lay(ay), self._lay(ax)
        B, C = out.shape[:2]
        e = ly.blends[rb] if rb > 0 else 0
        grid3 = []
        off = 0
        for k, per_k in enumerate(tiles3):
            grid = []
            if halo is not None and e:
                band = []
                for w in lx.extents:
                    shape = (B, C) + ((lt.extents[k],) if lt else ()) + (e, w)
                    n = int(np.prod(shape))
                    band.append(halo[off:off + n].view(shape))
                    off += n
                grid.append(band)
            grid += list(per_k)
            grid3.append([[t.numpy().view(np.uint16) for t in r] for r in grid])
        local_y = _local_axis(ly, rb, re_, e if halo is not None else 0)
        res = oracle_stitch(grid3, (lt, local_y, lx), "bf16") if lt else oracle_stitch(grid3[0], (local_y, lx), "bf16")
        res = res[..., local_y.kept[0] if (halo is not None and e) else 0:, :]
        out.copy_(torch.from_numpy(np.ascontiguousarray(res).view(np.int16)))
        return out

    def tb_stitch2d_shard(self, tiles, halo, ay, ax, rb, re_, out):
        return self._shard([tiles], halo, None, ay, ax, rb, re_, out)

    def tb_stitch3d_shard(self, tiles, halo, at, ay, ax, rb, re_, out):
        return self._shard(tiles, halo, at, ay, ax, rb, re_, out)

    def tb_stitch_shard_frames_layout(self, *args):
        return self.tb.tb_stitch_shard_frames_layout(*args)

    def tb_stitch_halo_pack_frames(self, frame_tiles, at, ay, ax, k, halo):
        e = self._lay(at).blends[k + 1]
        halo.copy_(torch.cat([t[:, :, -e:].reshape(-1) for row in frame_tiles for t in row]))

    def tb_stitch3d_shard_frames(self, tiles, halo, at, ay, ax, fb, fe, out):
        import numpy as np
        from oracle.stitch import stitch as oracle_stitch
        lt, ly, lx = self._lay(at), self._lay(ay), self._lay(ax)
        B, C = out.shape[:2]
        e = lt.blends[fb] if fb > 0 else 0
        grid3 = []
        if halo is not None and e:
            off, plane = 0, []
            for h in ly.extents:
                row = []
                for w in lx.extents:
                    shape = (B, C, e, h, w)
                    n = int(np.prod(shape))
                    row.append(halo[off:off + n].view(shape))
                    off += n
                plane.append(row)
            grid3.append(plane)
        grid3 += list(tiles)
        raw = [[[t.numpy().view(np.uint16) for t in r] for r in pl] for pl in grid3]
        local_t = _local_axis(lt, fb, fe, e if halo is not None else 0)
        res = oracle_stitch(raw, (local_t, ly, lx), "bf16")
        res = res[:, :, local_t.kept[0] if (halo is not None and e) else 0:]
        out.copy_(torch.from_numpy(np.ascontiguousarray(res).view(np.int16)))
        return out

    def new_partials(self, P, N, G, device=None):
        return torch.zeros((P, N, G, 8, 2), dtype=torch.int64)

    def tb_patch_gn_stats(self, patches, G, partials):
        # one record per unit: (count, mean, M2) of the patch's group elements
        import numpy as np
        for p, patch in enumerate(patches):
            partials[p] = _records(patch.double().numpy(), G, 1)[0]

    def tb_patch_gn_apply_gathered(self, patches, outs, G, every, R, gamma, beta, eps, silu):
        import numpy as np
        rec = every.numpy()
        c = rec[..., 0].astype(np.float64)
        mv = np.ascontiguousarray(rec[..., 1]).view(np.float32).reshape(rec.shape[:-1] + (2,)).astype(np.float64)
        n = c.sum(axis=(0, 3))
        mu = (c * mv[..., 0]).sum(axis=(0, 3)) / n
        var = (mv[..., 1] + c * (mv[..., 0] - mu[None, :, :, None]) ** 2).sum(axis=(0, 3)) / n
        for x, o in zip(patches, outs):
            xd = x.double().numpy()
            N, C = xd.shape[:2]
            cg = C // G
            y = np.empty_like(xd)
            for i in range(N):
                for ch in range(C):
                    g = ch // cg
                    z = (xd[i, ch] - mu[i, g]) / np.sqrt(var[i, g] + eps) * float(gamma[ch]) + float(beta[ch])
                    y[i, ch] = z / (1.0 + np.exp(-z)) if silu else z
            o.copy_(torch.from_numpy(y))
        return outs


def _stitch_share(tb, sharded, case, world, rank):
    # this rank's tile rows through the module's own entry point
    at, ay, ax, B, C = STITCH_CASES[case]
    lt, ly, lx, B, C, tiles = _stitch_tiles(case)
    a_t, a_y, a_x = (tb.Axis(*at) if at else None), tb.Axis(*ay), tb.Axis(*ax)
    lay = tb.tb_stitch_shard_layout(a_t, a_y, a_x, B, C, world, rank)
    rb, re_ = lay.row_begin, lay.row_end
    lib = _OracleLib(tb)
    if at:
        out = torch.empty((B, C, lt.out_extent, lay.out_rows, lx.out_extent), dtype=torch.int16)
        sharded.stitch3d_row_sharded([per_k[rb:re_] for per_k in tiles], a_t, a_y, a_x, out, lib=lib)
    else:
        out = torch.empty((B, C, lay.out_rows, lx.out_extent), dtype=torch.int16)
        sharded.stitch2d_row_sharded(tiles[0][rb:re_], a_y, a_x, out, lib=lib)
    return lay.out_row_begin, lay.out_rows, (out.numpy().view("uint16") if lay.out_rows else None)


def _frame_share(tb, sharded, world, rank):
    # the video case sharded along the time axis, through the module
    at, ay, ax, B, C = STITCH_CASES["video"]
    lt, ly, lx, B, C, tiles = _stitch_tiles("video")
    a_t, a_y, a_x = tb.Axis(*at), tb.Axis(*ay), tb.Axis(*ax)
    lay = tb.tb_stitch_shard_frames_layout(a_t, a_y, a_x, B, C, world, rank)
    out = torch.empty((B, C, lay.out_rows, ly.out_extent, lx.out_extent), dtype=torch.int16)
    sharded.stitch3d_frame_sharded(tiles[lay.row_begin:lay.row_end], a_t, a_y, a_x, out, lib=_OracleLib(tb))
    return lay.out_row_begin, lay.out_rows, (out.numpy().view("uint16") if lay.out_rows else None)


def _stitch_rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    from patch_groupnorm_gb300 import build
    build.build()
    from patch_groupnorm_gb300 import sharded, tileblend as tb
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = {case: _stitch_share(tb, sharded, case, world, rank) for case in STITCH_CASES}
        got["video_frames"] = _frame_share(tb, sharded, world, rank)
        q.put((rank, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_row_sharded_stitch_over_gloo_equals_the_unsharded_oracle(world):
    import numpy as np
    from oracle.stitch import stitch as oracle_stitch
    got = _spawn(_stitch_rank, world)
    for case in STITCH_CASES:
        lt, ly, lx, B, C, tiles = _stitch_tiles(case)
        raw = [[[t.numpy().view(np.uint16) for t in row] for row in per_k] for per_k in tiles]
        ref = oracle_stitch(raw, (lt, ly, lx), "bf16") if lt else oracle_stitch(raw[0], (ly, lx), "bf16")
        parts = [got[r][case] for r in range(world)]
        assert sum(p[1] for p in parts) == ly.out_extent, case
        assert [p[0] for p in parts] == [sum(p[1] for p in parts[:r]) for r in range(world)], case
        whole = np.concatenate([p[2] for p in parts if p[1] > 0], axis=-2)
        assert np.array_equal(whole, ref), case
    # the video, sharded along the frames instead
    lt, ly, lx, B, C, tiles = _stitch_tiles("video")
    raw = [[[t.numpy().view(np.uint16) for t in row] for row in per_k] for per_k in tiles]
    ref = oracle_stitch(raw, (lt, ly, lx), "bf16")
    parts = [got[r]["video_frames"] for r in range(world)]
    assert sum(p[1] for p in parts) == lt.out_extent
    assert np.array_equal(np.concatenate([p[2] for p in parts if p[1] > 0], axis=2), ref)


# --------------------------------------------------------------------------
# sharded PatchGroupNorm: records in the library's layout, gathered by the
# module's all-gather, pooled to the unsharded statistics
# --------------------------------------------------------------------------

def _records(patch, G, parts):
    """The library's record layout [1, N, G, TB_GN_PARTS, 2] (int64 count;
    fp32 mean and M2 packed in the second word) for one patch, each unit cut
    into `parts` contiguous parts; unused records have count 0."""
    import numpy as np
    N, C = patch.shape[:2]
    cg = C // G
    rec = np.zeros((1, N, G, 8, 2), dtype=np.int64)
    for n in range(N):
        for g in range(G):
            x = patch[n, g * cg:(g + 1) * cg].reshape(-1)
            for k, piece in enumerate(np.array_split(x, parts)):
                if piece.size == 0:
                    continue
                mu = piece.mean()
                rec[0, n, g, k, 0] = piece.size
                rec[0, n, g, k, 1] = np.array([mu, ((piece - mu) ** 2).sum()], dtype=np.float32).view(np.int64)[0]
    return torch.from_numpy(rec)


def _gn_rank(rank, world, port, q):
    # Every rank holds one patch; patch_group_norm_sharded writes its records
    # (cut into a rank-dependent number of parts, as GPUs with other SM counts
    # would), gathers every rank's records in one all-gather and normalises
    # its own patch with the pooled statistics; the result must be the
    # unsharded GroupNorm's patch.
    sys.path.insert(0, ROOT)
    import numpy as np
    from oracle import groupnorm as GN
    from patch_groupnorm_gb300 import build
    build.build()
    from patch_groupnorm_gb300 import sharded, tileblend as tb
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(3)
        x = rng.standard_normal((2, 12, 10, 14)) * 1.5
        sizes = [4, 3, 3][:world]                     # ragged height bands
        starts = np.cumsum([0] + sizes[:-1])
        patches = [x[:, :, s:s + n] + (r - 1) * 2.0 for r, (s, n) in enumerate(zip(starts, sizes))]
        gamma = 1.0 + 0.1 * rng.standard_normal(12)
        beta = 0.1 * rng.standard_normal(12)

        class Lib(_OracleLib):
            def tb_patch_gn_stats(self, ps, G, partials):
                for p_, patch in enumerate(ps):
                    partials[p_] = _records(patch.double().numpy(), G, 1 + 3 * rank)[0]

        mine = torch.from_numpy(patches[rank].copy())
        out = sharded.patch_group_norm_sharded([mine], 4, torch.from_numpy(gamma), torch.from_numpy(beta), 1e-6,
                                               silu=True, lib=Lib(tb))[0]
        want = GN.patch_group_norm(patches, 4, gamma, beta, 1e-6, silu=True)[rank]
        q.put((rank, bool(np.abs(out.numpy() - want).max() < 1e-5)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_sharded_groupnorm_over_gloo_equals_the_unsharded_oracle():
    assert _spawn(_gn_rank, 3) == {r: True for r in range(3)}
