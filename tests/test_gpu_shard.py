"""GPU parity of the sharded paths, with the ranks run one after another on
one GPU (every call through the C ABI):

* row-sharded stitch: each rank packs the band its last tile row lends to the
  next rank (tb_stitch_halo_pack), the next rank stitches its own tile rows
  with that band (tb_stitch2d_shard / tb_stitch3d_shard); the ranks' outputs
  concatenated along the height equal the CPU oracle's unsharded stitch bit
  for bit, at every workload's full size and on small random grids;
* sharded PatchGroupNorm: each patch's statistics from its own call (as each
  rank computes them), the records concatenated (as an all-gather hands them
  over), and each patch normalised alone with the pooled statistics
  (tb_patch_gn_apply_gathered); within the GroupNorm tolerance of the float64
  oracle.
"""
import random

import numpy as np
import pytest
import torch

from oracle.geometry import axis_layout
from oracle.stitch import stitch as oracle_stitch
from patch_groupnorm_gb300 import synth
from patch_groupnorm_gb300 import workloads as W
from tests.stitch_helpers import TORCH, boxes, to_storage
from tests.tolerance import gn_violation

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tbl():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from patch_groupnorm_gb300 import build
    build.build()
    from patch_groupnorm_gb300 import tileblend
    return tileblend


def _axis(tbl, a):
    return tbl.Axis(a.latent_extent, a.latent_tile, a.overlap, a.scale)


def _storage_grid(tiles, dtype):
    if isinstance(tiles, torch.Tensor):
        return to_storage(tiles, dtype)
    return [_storage_grid(t, dtype) for t in tiles]


def _sharded_gpu(tbl, tiles_cpu, axes, dtype, B, C, world):
    """Every rank's share, run in rank order on one GPU; returns the ranks'
    outputs concatenated along the height."""
    ndim = len(axes)
    ta = [_axis(tbl, a) for a in axes]
    at, ay, ax = (None, ta[0], ta[1]) if ndim == 2 else ta
    lays = [axis_layout(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in axes]
    W_out = lays[-1].out_extent
    T_out = lays[0].out_extent if ndim == 3 else None
    if ndim == 2:
        dev = [[t.cuda() for t in row] for row in tiles_cpu]
    else:
        dev = [[[t.cuda() for t in row] for row in pl] for pl in tiles_cpu]
    outs, bands = [], {}
    for r in range(world):
        lay = tbl.tb_stitch_shard_layout(at, ay, ax, B, C, world, r)
        rb, re_ = lay.row_begin, lay.row_end
        if ndim == 2:
            mine = dev[rb:re_]
            out = torch.full((B, C, lay.out_rows, W_out), float("nan"), dtype=TORCH[dtype], device="cuda")
        else:
            mine = [pl[rb:re_] for pl in dev]
            out = torch.full((B, C, T_out, lay.out_rows, W_out), float("nan"), dtype=TORCH[dtype], device="cuda")
        halo = bands.get(r)
        assert (halo is None) == (lay.halo_elems == 0)
        if halo is not None:
            assert halo.numel() == lay.halo_elems
        if ndim == 2:
            tbl.tb_stitch2d_shard(mine, halo, ay, ax, rb, re_, out)
        else:
            tbl.tb_stitch3d_shard(mine, halo, at, ay, ax, rb, re_, out)
        if lay.send_elems:
            send = torch.empty(lay.send_elems, dtype=TORCH[dtype], device="cuda")
            row = mine[-1] if ndim == 2 else [pl[-1] for pl in mine]
            tbl.tb_stitch_halo_pack(row, at, ay, ax, re_ - 1, send)
            bands[r + 1] = send
        outs.append(out)
    torch.cuda.synchronize()
    return torch.cat([o.cpu() for o in outs], dim=-2)


def _check_equal(got: torch.Tensor, ref: np.ndarray, dtype: str):
    g = to_storage(got, dtype)
    assert g.shape == ref.shape
    if not np.array_equal(g, ref):
        bad = np.argwhere(g != ref)
        raise AssertionError("%d of %d elements differ; first at %s" % (len(bad), ref.size, tuple(bad[0])))


@pytest.mark.parametrize("name", ["image_1024_f32", "image_2048_bf16", "wide_1600x2048_bf16",
                                  "video_49x480x832_bf16"])
def test_full_workload_sharded_bit_exact(tbl, name):
    w = W.STITCH[name]
    lays = [axis_layout(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in w.axes]
    tiles = W.make_stitch_tiles(w, [boxes(l, a.scale) for l, a in zip(lays, w.axes)], [l.out_extent for l in lays])
    ref = oracle_stitch(_storage_grid(tiles, w.dtype), lays, w.dtype)
    n_rows = lays[-2].n
    for world in sorted({2, 3, n_rows, n_rows + 2}):
        _check_equal(_sharded_gpu(tbl, tiles, w.axes, w.dtype, w.B, w.C, world), ref, w.dtype)


def test_halo_pack_is_the_bottom_band_of_each_tile(tbl):
    w = W.STITCH["video_49x480x832_bf16"]
    axes = [_axis(tbl, a) for a in w.axes]
    lays = [tbl.tb_axis_layout(a) for a in axes]
    rng = np.random.default_rng(11)
    row = 0                                      # rank 0 of 3 holds tile row 0 and sends its band
    e = lays[1].blends[row + 1]
    tiles = [[torch.from_numpy(rng.uniform(-1, 1, (1, 3, lt, lays[1].extents[row], lx))).to(torch.bfloat16).cuda()
              for lx in lays[2].extents] for lt in lays[0].extents]
    lay = tbl.tb_stitch_shard_layout(*axes, 1, 3, 3, 0)
    send = torch.empty(lay.send_elems, dtype=torch.bfloat16, device="cuda")
    tbl.tb_stitch_halo_pack(tiles, *axes, row, send)
    want = torch.cat([t[:, :, :, -e:, :].reshape(-1) for per_k in tiles for t in per_k])
    torch.cuda.synchronize()
    assert torch.equal(send.view(torch.int16), want.view(torch.int16))


def _random_axes(rnd, ndim):
    axes = []
    for a in range(ndim):
        while True:
            tile = rnd.randint(2, 24)
            ov = rnd.choice([0.0, 0.125, 0.25, 1 / 3, 0.5])
            stride = int(tile * (1 - ov))
            if stride < 1:
                continue
            scale = 1 if (ndim == 3 and a == 0) else rnd.choice([1, 2, 4, 8])
            ext = rnd.randint(1, 6 * stride)
            lay = axis_layout(ext, tile, ov, scale)
            ok = all(lay.extents[k] >= lay.blends[k] + lay.blends[k + 1] for k in range(1, lay.n - 1))
            if ok and lay.n <= 6:
                axes.append(W.AxisSpec(ext, tile, ov, scale))
                break
    return axes


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("ndim", [2, 3])
def test_random_small_grids_sharded_bit_exact(tbl, dtype, ndim):
    rnd = random.Random(300 * ndim + len(dtype))
    rng = np.random.default_rng(ndim + 40)
    for trial in range(16 if ndim == 2 else 8):
        axes = _random_axes(rnd, ndim)
        lays = [axis_layout(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in axes]
        B, C = rnd.randint(1, 2), rnd.randint(1, 3)
        if ndim == 2:
            tiles = [[torch.from_numpy(rng.uniform(-1, 1, (B, C, ly, lx))).to(TORCH[dtype])
                      for lx in lays[1].extents] for ly in lays[0].extents]
        else:
            tiles = [[[torch.from_numpy(rng.uniform(-1, 1, (B, C, lt, ly, lx))).to(TORCH[dtype])
                       for lx in lays[2].extents] for ly in lays[1].extents] for lt in lays[0].extents]
        ref = oracle_stitch(_storage_grid(tiles, dtype), lays, dtype)
        for world in (2, 3, 5):
            _check_equal(_sharded_gpu(tbl, tiles, axes, dtype, B, C, world), ref, dtype)


def test_shard_matches_the_library_unsharded_stitch(tbl):
    w = W.STITCH["image_2048_bf16_uniform"]
    axes = [_axis(tbl, a) for a in w.axes]
    lays = [tbl.tb_axis_layout(a) for a in axes]
    tiles = W.make_stitch_tiles(w, [list(zip(l.origins, l.extents)) for l in lays], [l.out_extent for l in lays])
    full = torch.empty((w.B, w.C, lays[0].out_extent, lays[1].out_extent), dtype=torch.bfloat16, device="cuda")
    tbl.tb_stitch2d([[t.cuda() for t in row] for row in tiles], axes[0], axes[1], full)
    got = _sharded_gpu(tbl, tiles, w.axes, w.dtype, w.B, w.C, 4)
    assert torch.equal(got.view(torch.int16), full.cpu().view(torch.int16))


def test_shard_rejects_a_missing_band_and_a_wrong_row_count(tbl):
    ay, ax = tbl.Axis(128, 64, 0.25, 8), tbl.Axis(64, 64, 0.25, 8)
    lay = tbl.tb_stitch_shard_layout(None, ay, ax, 1, 1, 2, 1)
    tiles = [[torch.zeros((1, 1, 512, 512), dtype=torch.bfloat16, device="cuda")] for _ in range(lay.row_end -
                                                                                                  lay.row_begin)]
    out = torch.empty((1, 1, lay.out_rows, 512), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tbl.TileBlendError) as e:
        tbl.tb_stitch2d_shard(tiles, None, ay, ax, lay.row_begin, lay.row_end, out)
    assert e.value.status == tbl.TB_ERR_NULL
    bad = torch.empty((1, 1, lay.out_rows + 1, 512), dtype=torch.bfloat16, device="cuda")
    halo = torch.zeros(lay.halo_elems, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tbl.TileBlendError) as e:
        tbl.tb_stitch2d_shard(tiles, halo, ay, ax, lay.row_begin, lay.row_end, bad)
    assert e.value.status == tbl.TB_ERR_SHAPE


# --------------------------------------------------------------------------
# sharded PatchGroupNorm: per-rank statistics, gathered records, local apply
# --------------------------------------------------------------------------

def _rank_records(tbl, patches, G, groups_of_patches):
    """Statistics of each group of patches from its own call (a rank's call);
    the record sets concatenated in patch order, as an all-gather returns
    them."""
    sets = []
    for idx in groups_of_patches:
        part = tbl.new_partials(len(idx), patches[0].shape[0], G)
        tbl.tb_patch_gn_stats([patches[i] for i in idx], G, part)
        sets.append(part)
    return torch.cat(sets, dim=0)


@pytest.mark.parametrize("name", list(W.GROUPNORM))
def test_per_rank_statistics_and_local_apply_full_workload(tbl, name):
    w = W.GROUPNORM[name]
    patches, gamma, beta = W.make_groupnorm_inputs(w)
    dev = [p.cuda() for p in patches]
    g, b = gamma.cuda(), beta.cuda()
    P = len(dev)
    every = _rank_records(tbl, dev, w.groups, [[p] for p in range(P)])
    outs = []
    for p in range(P):          # each rank normalises only its own patch
        o = torch.empty_like(dev[p])
        tbl.tb_patch_gn_apply_gathered([dev[p]], [o], w.groups, every, P, g, b, w.eps, True)
        outs.append(o)
    torch.cuda.synchronize()
    with np.errstate(over="ignore"):
        assert gn_violation([o.cpu() for o in outs], patches, gamma, beta, w.groups, w.eps, True, w.dtype) <= 1.0


def test_records_from_calls_that_split_differently_combine(tbl):
    # one call over patches 0-2 and one for patch 3: the calls cut their units
    # into pieces of different sizes (a call's split depends on its total
    # size); the records describe themselves
    patches, gamma, beta = synth.groupnorm_patches(31, (2, 64, 256, 256), 2, 4, (-3.0, -1.0, 1.0, 3.0), "bf16")
    dev = [p.cuda() for p in patches]
    every = _rank_records(tbl, dev, 16, [[0, 1, 2], [3]])
    counts = every[..., 0]                           # elements per record
    assert counts[:3].max() != counts[3:].max()
    outs = [torch.empty_like(p) for p in dev]
    tbl.tb_patch_gn_apply(dev, outs, 16, every, gamma.cuda(), beta.cuda(), 1e-6, True)
    local = [torch.empty_like(dev[2])]
    tbl.tb_patch_gn_apply_gathered([dev[2]], local, 16, every, 4, gamma.cuda(), beta.cuda(), 1e-6, True)
    torch.cuda.synchronize()
    assert torch.equal(local[0], outs[2])
    with np.errstate(over="ignore"):
        assert gn_violation([o.cpu() for o in outs], patches, gamma, beta, 16, 1e-6, True, "bf16") <= 1.0


def test_gathered_apply_with_empty_records_and_record_order(tbl):
    # a rank with an empty patch contributes count-0 records only; the order
    # of the record sets does not change the pooled statistics' elements
    patches, gamma, beta = synth.groupnorm_patches(32, (1, 32, 30, 16), 2, 3, (-2.0, 0.0, 2.0), "f32")
    empty = torch.empty((1, 32, 0, 16), dtype=torch.float32)
    dev = [p.cuda() for p in patches] + [empty.cuda()]
    every = _rank_records(tbl, dev, 8, [[3], [2], [0], [1]])
    assert (every[0, ..., 0] == 0).all()
    outs = [torch.empty_like(p) for p in dev[:3]]
    for p in range(3):
        tbl.tb_patch_gn_apply_gathered([dev[p]], [outs[p]], 8, every, 4, gamma.cuda(), beta.cuda(), 1e-6, True)
    torch.cuda.synchronize()
    assert gn_violation([o.cpu() for o in outs], patches, gamma, beta, 8, 1e-6, True, "f32") <= 1.0


def test_sharded_module_on_a_one_rank_nccl_group(tbl):
    # the multi-rank module itself on a GPU: one rank, so the stitch needs no
    # band and the all-gather returns the rank's own records; results equal
    # the direct library calls bit for bit
    import socket
    import torch.distributed as dist
    from patch_groupnorm_gb300 import sharded
    sk = socket.socket()
    sk.bind(("127.0.0.1", 0))
    port = sk.getsockname()[1]
    sk.close()
    dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % port, rank=0, world_size=1)
    try:
        w = W.STITCH["image_2048_bf16_uniform"]
        axes = [_axis(tbl, a) for a in w.axes]
        lays = [tbl.tb_axis_layout(a) for a in axes]
        tiles = W.make_stitch_tiles(w, [list(zip(l.origins, l.extents)) for l in lays],
                                    [l.out_extent for l in lays])
        dev = [[t.cuda() for t in row] for row in tiles]
        shape = (w.B, w.C, lays[0].out_extent, lays[1].out_extent)
        want = tbl.tb_stitch2d(dev, axes[0], axes[1], torch.empty(shape, dtype=torch.bfloat16, device="cuda"))
        got = sharded.stitch2d_row_sharded(dev, axes[0], axes[1], torch.empty_like(want))
        patches, gamma, beta = synth.groupnorm_patches(33, (1, 64, 32, 48), 2, 2, (-2.0, 2.0), "bf16")
        dp = [p.cuda() for p in patches]
        ref = tbl.patch_group_norm(dp, 16, gamma.cuda(), beta.cuda(), 1e-6, silu=True)
        outs = sharded.patch_group_norm_sharded(dp, 16, gamma.cuda(), beta.cuda(), 1e-6, silu=True)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
        for o, r in zip(outs, ref):
            assert torch.equal(o.view(torch.int16), r.view(torch.int16))
    finally:
        dist.destroy_process_group()


# --------------------------------------------------------------------------
# frame-sharded video stitch
# --------------------------------------------------------------------------

def _frame_sharded_gpu(tbl, tiles_cpu, axes, dtype, B, C, world):
    """Every rank's frame tiles, run in rank order on one GPU; returns the
    ranks' outputs concatenated along the frames."""
    at, ay, ax = [_axis(tbl, a) for a in axes]
    lays = [axis_layout(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in axes]
    dev = [[[t.cuda() for t in row] for row in pl] for pl in tiles_cpu]
    outs, bands = [], {}
    for r in range(world):
        lay = tbl.tb_stitch_shard_frames_layout(at, ay, ax, B, C, world, r)
        mine = dev[lay.row_begin:lay.row_end]
        out = torch.full((B, C, lay.out_rows, lays[1].out_extent, lays[2].out_extent), float("nan"),
                         dtype=TORCH[dtype], device="cuda")
        halo = bands.get(r)
        assert (halo is None) == (lay.halo_elems == 0)
        tbl.tb_stitch3d_shard_frames(mine, halo, at, ay, ax, lay.row_begin, lay.row_end, out)
        if lay.send_elems:
            send = torch.empty(lay.send_elems, dtype=TORCH[dtype], device="cuda")
            tbl.tb_stitch_halo_pack_frames(mine[-1], at, ay, ax, lay.row_end - 1, send)
            bands[r + 1] = send
        outs.append(out)
    torch.cuda.synchronize()
    return torch.cat([o.cpu() for o in outs], dim=2)


def test_full_video_frame_sharded_bit_exact(tbl):
    w = W.STITCH["video_49x480x832_bf16"]
    lays = [axis_layout(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in w.axes]
    tiles = W.make_stitch_tiles(w, [boxes(l, a.scale) for l, a in zip(lays, w.axes)], [l.out_extent for l in lays])
    ref = oracle_stitch(_storage_grid(tiles, w.dtype), lays, w.dtype)
    for world in (2, 3, lays[0].n, lays[0].n + 2):
        _check_equal(_frame_sharded_gpu(tbl, tiles, w.axes, w.dtype, w.B, w.C, world), ref, w.dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_random_small_videos_frame_sharded_bit_exact(tbl, dtype):
    rnd = random.Random(77 + len(dtype))
    rng = np.random.default_rng(78)
    for trial in range(8):
        axes = _random_axes(rnd, 3)
        lays = [axis_layout(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in axes]
        B, C = rnd.randint(1, 2), rnd.randint(1, 3)
        tiles = [[[torch.from_numpy(rng.uniform(-1, 1, (B, C, lt, ly, lx))).to(TORCH[dtype])
                   for lx in lays[2].extents] for ly in lays[1].extents] for lt in lays[0].extents]
        ref = oracle_stitch(_storage_grid(tiles, dtype), lays, dtype)
        for world in (2, 3):
            _check_equal(_frame_sharded_gpu(tbl, tiles, axes, dtype, B, C, world), ref, dtype)


def test_frame_halo_pack_is_the_last_frames_of_each_tile(tbl):
    w = W.STITCH["video_49x480x832_bf16"]
    at, ay, ax = [_axis(tbl, a) for a in w.axes]
    lays = [tbl.tb_axis_layout(a) for a in (at, ay, ax)]
    rng = np.random.default_rng(12)
    k = 1
    e = lays[0].blends[k + 1]
    tiles = [[torch.from_numpy(rng.uniform(-1, 1, (1, 3, lays[0].extents[k], ly, lx))).to(torch.bfloat16).cuda()
              for lx in lays[2].extents] for ly in lays[1].extents]
    lay = tbl.tb_stitch_shard_frames_layout(at, ay, ax, 1, 3, 5, k)
    send = torch.empty(lay.send_elems, dtype=torch.bfloat16, device="cuda")
    tbl.tb_stitch_halo_pack_frames(tiles, at, ay, ax, k, send)
    want = torch.cat([t[:, :, -e:].reshape(-1) for row in tiles for t in row])
    torch.cuda.synchronize()
    assert torch.equal(send.view(torch.int16), want.view(torch.int16))
