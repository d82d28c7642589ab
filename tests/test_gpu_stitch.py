"""GPU parity of tb_stitch2d / tb_stitch3d against the CPU oracle: bit-exact
on every element, at the full workload sizes and on small random grids that
span several tiles, ragged slivers, both the 16-byte and the per-element
kernel paths, and the degenerate cases."""
import itertools
import random

import numpy as np
import pytest
import torch

from oracle.geometry import axis_layout
from oracle.stitch import stitch as oracle_stitch
from patch_groupnorm_gb300 import workloads as W
from tests.stitch_helpers import TORCH, boxes, to_storage

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


def _oracle_layouts(axes):
    return [axis_layout(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in axes]


def _storage_grid(tiles, dtype):
    if isinstance(tiles, torch.Tensor):
        return to_storage(tiles, dtype)
    return [_storage_grid(t, dtype) for t in tiles]


def _to_cuda(tiles):
    if isinstance(tiles, torch.Tensor):
        return tiles.cuda()
    return [_to_cuda(t) for t in tiles]


def _run_gpu(tbl, tiles_cpu, axes, dtype, B, C, offset_elems=0):
    """Stitch on the GPU; with offset_elems > 0 every tensor starts that many
    elements into a larger buffer (misaligned for the 16-byte path)."""
    lays = _oracle_layouts(axes)
    out_shape = (B, C) + tuple(l.out_extent for l in lays)
    keep = []

    def place(t):
        if offset_elems == 0:
            return t.cuda()
        buf = torch.empty(t.numel() + offset_elems, dtype=t.dtype, device="cuda")
        v = buf[offset_elems:].view(t.shape)
        v.copy_(t)
        keep.append(buf)
        return v

    def walk(x):
        return place(x) if isinstance(x, torch.Tensor) else [walk(y) for y in x]

    tiles = walk(tiles_cpu)
    if offset_elems:
        ob = torch.empty(int(np.prod(out_shape)) + offset_elems, dtype=TORCH[dtype], device="cuda")
        out = ob[offset_elems:].view(out_shape)
    else:
        out = torch.empty(out_shape, dtype=TORCH[dtype], device="cuda")
    if len(axes) == 2:
        tbl.tb_stitch2d(tiles, _axis(tbl, axes[0]), _axis(tbl, axes[1]), out)
    else:
        tbl.tb_stitch3d(tiles, _axis(tbl, axes[0]), _axis(tbl, axes[1]), _axis(tbl, axes[2]), out)
    torch.cuda.synchronize()
    return out.cpu()


def _check_equal(got: torch.Tensor, ref: np.ndarray, dtype: str):
    g = to_storage(got, dtype)
    if not np.array_equal(g, ref):
        bad = np.argwhere(g != ref)
        raise AssertionError("%d of %d elements differ; first at %s: got %r want %r" % (
            len(bad), ref.size, tuple(bad[0]), g[tuple(bad[0])], ref[tuple(bad[0])]))


# --------------------------------------------------------------------------
# full workloads
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", list(W.STITCH))
def test_full_workload_bit_exact(tbl, name):
    w = W.STITCH[name]
    lays = _oracle_layouts(w.axes)
    bx = [boxes(l, a.scale) for l, a in zip(lays, w.axes)]
    tiles = W.make_stitch_tiles(w, bx, [l.out_extent for l in lays])
    ref = oracle_stitch(_storage_grid(tiles, w.dtype), lays, w.dtype)
    got = _run_gpu(tbl, tiles, w.axes, w.dtype, w.B, w.C)
    _check_equal(got, ref, w.dtype)


def test_full_workload_repeatable(tbl):
    w = W.STITCH["image_2048_bf16_uniform"]
    lays = _oracle_layouts(w.axes)
    tiles = W.make_stitch_tiles(w, [boxes(l, a.scale) for l, a in zip(lays, w.axes)], [l.out_extent for l in lays])
    a = _run_gpu(tbl, tiles, w.axes, w.dtype, w.B, w.C)
    b = _run_gpu(tbl, tiles, w.axes, w.dtype, w.B, w.C)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# --------------------------------------------------------------------------
# small random grids: several tiles, ragged slivers, both kernel paths
# --------------------------------------------------------------------------

def _random_case(rnd, ndim):
    axes = []
    for a in range(ndim):
        while True:
            tile = rnd.randint(2, 24)
            ov = rnd.choice([0.0, 0.125, 0.25, 0.25, 1 / 3, 0.5])
            stride = int(tile * (1 - ov))
            if stride < 1:
                continue
            scale = 1 if (ndim == 3 and a == 0) else rnd.choice([1, 2, 4, 8])
            ext = rnd.randint(1, 5 * stride)
            lay = axis_layout(ext, tile, ov, scale)
            ok = all(lay.extents[k] >= lay.blends[k] + lay.blends[k + 1] for k in range(1, lay.n - 1))
            if ok and lay.n <= 6:
                axes.append(W.AxisSpec(ext, tile, ov, scale))
                break
    return axes


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("ndim", [2, 3])
def test_random_small_grids_bit_exact(tbl, dtype, ndim):
    rnd = random.Random(100 * ndim + len(dtype))
    rng = np.random.default_rng(ndim)
    for trial in range(25 if ndim == 2 else 12):
        axes = _random_case(rnd, ndim)
        lays = _oracle_layouts(axes)
        B, C = rnd.randint(1, 2), rnd.randint(1, 3)
        if ndim == 2:
            tiles = [[torch.from_numpy(rng.uniform(-1, 1, (B, C, ly, lx))).to(TORCH[dtype])
                      for lx in lays[1].extents] for ly in lays[0].extents]
        else:
            tiles = [[[torch.from_numpy(rng.uniform(-1, 1, (B, C, lt, ly, lx))).to(TORCH[dtype])
                       for lx in lays[2].extents] for ly in lays[1].extents] for lt in lays[0].extents]
        ref = oracle_stitch(_storage_grid(tiles, dtype), lays, dtype)
        got = _run_gpu(tbl, tiles, axes, dtype, B, C)
        _check_equal(got, ref, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_vector_path_geometry_spanning_tiles(tbl, dtype):
    # 8-aligned widths so the 16-byte path runs, several tiles and a ragged
    # last tile on both axes, a wider-than-512-chunk row (row segments)
    axes = [W.AxisSpec(21, 16, 0.25, 8), W.AxisSpec(1100, 64, 0.25, 8)]
    lays = _oracle_layouts(axes)
    rng = np.random.default_rng(5)
    tiles = [[torch.from_numpy(rng.uniform(-1, 1, (1, 2, ly, lx))).to(TORCH[dtype])
              for lx in lays[1].extents] for ly in lays[0].extents]
    ref = oracle_stitch(_storage_grid(tiles, dtype), lays, dtype)
    _check_equal(_run_gpu(tbl, tiles, axes, dtype, 1, 2), ref, dtype)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_misaligned_pointers_take_the_element_path(tbl, dtype):
    w = W.STITCH["image_1024_f32"]
    axes = [W.AxisSpec(40, 16, 0.25, 8), W.AxisSpec(40, 16, 0.25, 8)]
    lays = _oracle_layouts(axes)
    rng = np.random.default_rng(6)
    tiles = [[torch.from_numpy(rng.uniform(-1, 1, (2, 3, ly, lx))).to(TORCH[dtype])
              for lx in lays[1].extents] for ly in lays[0].extents]
    ref = oracle_stitch(_storage_grid(tiles, dtype), lays, dtype)
    _check_equal(_run_gpu(tbl, tiles, axes, dtype, 2, 3, offset_elems=1), ref, dtype)


# --------------------------------------------------------------------------
# degenerate cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_tile_and_zero_overlap(tbl, dtype):
    rng = np.random.default_rng(7)
    for axes in ([W.AxisSpec(30, 64, 0.25, 8), W.AxisSpec(20, 64, 0.25, 8)],     # one tile
                 [W.AxisSpec(30, 8, 0.0, 8), W.AxisSpec(20, 8, 0.0, 4)]):        # no overlap
        lays = _oracle_layouts(axes)
        tiles = [[torch.from_numpy(rng.uniform(-1, 1, (1, 3, ly, lx))).to(TORCH[dtype])
                  for lx in lays[1].extents] for ly in lays[0].extents]
        ref = oracle_stitch(_storage_grid(tiles, dtype), lays, dtype)
        _check_equal(_run_gpu(tbl, tiles, axes, dtype, 1, 3), ref, dtype)


def test_empty_batch_writes_nothing(tbl):
    ay = tbl.Axis(128, 64, 0.25, 8)
    lay = tbl.tb_axis_layout(ay)
    tiles = [[torch.empty((0, 3, ly, lx), device="cuda") for lx in lay.extents] for ly in lay.extents]
    out = torch.empty((0, 3, 1024, 1024), device="cuda")
    tbl.tb_stitch2d(tiles, ay, ay, out)
    torch.cuda.synchronize()


def test_output_guard_bands_untouched(tbl):
    # the output sits between two canary bands; nothing outside it changes
    w = W.STITCH["image_1024_f32"]
    lays = _oracle_layouts(w.axes)
    tiles = W.make_stitch_tiles(w, [boxes(l, a.scale) for l, a in zip(lays, w.axes)], [l.out_extent for l in lays])
    n = w.B * w.C * lays[0].out_extent * lays[1].out_extent
    guard = 4096
    buf = torch.full((n + 2 * guard,), 12345.0, device="cuda")
    out = buf[guard:guard + n].view(w.B, w.C, lays[0].out_extent, lays[1].out_extent)
    tbl.tb_stitch2d(_to_cuda(tiles), _axis(tbl, w.axes[0]), _axis(tbl, w.axes[1]), out)
    torch.cuda.synchronize()
    assert (buf[:guard] == 12345.0).all() and (buf[guard + n:] == 12345.0).all()
    ref = oracle_stitch(_storage_grid(tiles, "f32"), lays, "f32")
    _check_equal(out.cpu(), ref, "f32")


def test_tiles_are_not_modified(tbl):
    w = W.STITCH["wide_1600x2048_bf16"]
    lays = _oracle_layouts(w.axes)
    tiles = W.make_stitch_tiles(w, [boxes(l, a.scale) for l, a in zip(lays, w.axes)], [l.out_extent for l in lays])
    dev = _to_cuda(tiles)
    out = torch.empty((w.B, w.C, lays[0].out_extent, lays[1].out_extent), dtype=torch.bfloat16, device="cuda")
    tbl.tb_stitch2d(dev, _axis(tbl, w.axes[0]), _axis(tbl, w.axes[1]), out)
    torch.cuda.synchronize()
    for row_c, row_d in zip(tiles, dev):
        for tc, td in zip(row_c, row_d):
            assert torch.equal(tc.view(torch.int16), td.cpu().view(torch.int16))


def test_graph_capture_replays_with_new_inputs(tbl):
    # parameters travel by value, so a captured launch replays correctly when
    # the tile contents at the same addresses change
    w = W.STITCH["image_1024_f32"]
    lays = _oracle_layouts(w.axes)
    bx = [boxes(l, a.scale) for l, a in zip(lays, w.axes)]
    tiles0 = W.make_stitch_tiles(w, bx, [l.out_extent for l in lays])
    dev = _to_cuda(tiles0)
    out = torch.empty((w.B, w.C, lays[0].out_extent, lays[1].out_extent), device="cuda")
    ay, ax = _axis(tbl, w.axes[0]), _axis(tbl, w.axes[1])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tbl.tb_stitch2d(dev, ay, ax, out)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tbl.tb_stitch2d(dev, ay, ax, out)
    for seed in (11, 12, 13):
        w2 = W.StitchWorkload(w.name, w.dtype, w.B, w.C, w.axes, "uniform", seed)
        fresh = W.make_stitch_tiles(w2, bx, [l.out_extent for l in lays])
        for rd, rf in zip(dev, fresh):
            for td, tf in zip(rd, rf):
                td.copy_(tf)
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_stitch(_storage_grid(fresh, "f32"), lays, "f32")
        _check_equal(out.cpu(), ref, "f32")


@pytest.mark.parametrize("ndim", [2, 3])
def test_largest_tile_grid_bit_exact(tbl, ndim):
    # TB_MAX_TILES tiles in one call: 16 x 64 (2D) and 4 x 16 x 16 (3D) small
    # tiles, 64 along one axis (TB_MAX_TILES_PER_AXIS)
    if ndim == 2:
        axes = [W.AxisSpec(96, 8, 0.25, 1), W.AxisSpec(384, 8, 0.25, 1)]
    else:
        axes = [W.AxisSpec(24, 8, 0.25, 1), W.AxisSpec(96, 8, 0.25, 1), W.AxisSpec(96, 8, 0.25, 1)]
    lays = _oracle_layouts(axes)
    assert int(np.prod([l.n for l in lays])) == tbl.TB_MAX_TILES
    rng = np.random.default_rng(40 + ndim)
    if ndim == 2:
        tiles = [[torch.from_numpy(rng.uniform(-1, 1, (1, 2, ly, lx))).to(torch.bfloat16)
                  for lx in lays[1].extents] for ly in lays[0].extents]
    else:
        tiles = [[[torch.from_numpy(rng.uniform(-1, 1, (1, 2, lt, ly, lx))).to(torch.bfloat16)
                   for lx in lays[2].extents] for ly in lays[1].extents] for lt in lays[0].extents]
    ref = oracle_stitch(_storage_grid(tiles, "bf16"), lays, "bf16")
    _check_equal(_run_gpu(tbl, tiles, axes, "bf16", 1, 2), ref, "bf16")


def test_tall_wide_tiles_with_more_piece_ranks_than_the_rank_table(tbl):
    # 4096-row tiles 1536 px kept wide: a copy box one 16-byte chunk per
    # thread across gives 16-row pieces, 192 of them for one tile -- more
    # ranks than the one-dimensional grid's table holds -- on a grid larger
    # than one resident wave: the two-dimensional grid is used instead
    axes = [W.AxisSpec(512, 512, 0.25, 8), W.AxisSpec(256, 256, 0.25, 8)]
    lays = _oracle_layouts(axes)
    assert [l.extents for l in lays] == [[4096, 1024], [2048, 512]]
    rng = np.random.default_rng(192)
    tiles = [[torch.from_numpy(rng.uniform(-1, 1, (1, 3, ly, lx)).astype(np.float32)).to(torch.bfloat16)
              for lx in lays[1].extents] for ly in lays[0].extents]
    ref = oracle_stitch(_storage_grid(tiles, "bf16"), lays, "bf16")
    _check_equal(_run_gpu(tbl, tiles, axes, "bf16", 1, 3), ref, "bf16")


def test_no_kernel_reported_a_problem(tbl):
    # the device status word stays 0 through every stitch above (no copy
    # wait ran out, no bounds check fired)
    assert tbl.tb_device_status(clear=True) == tbl.TB_DEV_OK
