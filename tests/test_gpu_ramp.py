"""GPU parity of tb_stitch2d_ramp against the float64 oracle (oracle/ramp.py).

Tolerances (fp32 arithmetic, one rounding into storage):
  * fp16 / bf16: 1 ulp of the oracle's once-rounded value, taken at
    max(|value|, 2^-8), as for the GroupNorm output;
  * fp32: 4e-6 times the largest |tile value| (a handful of fp32 roundings
    in the weights and the sum of at most nine terms);
  * wherever exactly one tile has positive weight the output is that tile's
    value, bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle import rounding as R
from oracle.ramp import axis_weights, ramp_stitch_2d
from patch_groupnorm_gb300 import synth
from patch_groupnorm_gb300 import workloads as W
from tests.tolerance import violation
from tests.stitch_helpers import TORCH, to_storage

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tbl():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from patch_groupnorm_gb300 import build
    build.build()
    from patch_groupnorm_gb300 import tileblend
    return tileblend


def _run(tbl, tiles, ay, ax, dtype):
    B, C = tiles[0][0].shape[:2]
    out = torch.empty((B, C, ay.out_extent, ax.out_extent), dtype=TORCH[dtype], device="cuda")
    tbl.tb_stitch2d_ramp([[t.cuda() for t in row] for row in tiles], ay, ax, out)
    torch.cuda.synchronize()
    return out.cpu()


def _check(tbl, tiles, ay, ax, dtype):
    got = _run(tbl, tiles, ay, ax, dtype)
    tiles64 = [[t.double().numpy() for t in row] for row in tiles]
    exact = ramp_stitch_2d(tiles64, ay.origins, ax.origins, ay.tile_extent, ax.tile_extent,
                           (ay.out_extent, ax.out_extent), ay.zero, ay.ramp, ax.zero, ax.ramp)
    g = got.double().numpy()
    if dtype == "f32":
        scale = max(1.0, max(float(np.abs(t).max()) for row in tiles64 for t in row))
        assert np.abs(g - exact).max() <= 4e-6 * scale
    else:
        assert violation(g, exact, dtype) <= 1.0
    # single-cover samples are copies
    wy = axis_weights(ay.origins, ay.tile_extent, ay.out_extent, ay.zero, ay.ramp)
    wx = axis_weights(ax.origins, ax.tile_extent, ax.out_extent, ax.zero, ax.ramp)
    cy, cx = (wy > 0).sum(0), (wx > 0).sum(0)
    gs = to_storage(got, dtype)
    for i, oy in enumerate(ay.origins):
        for j, ox in enumerate(ax.origins):
            ys = [y for y in range(oy, oy + ay.tile_extent) if cy[y] == 1 and wy[i, y] > 0]
            xs = [x for x in range(ox, ox + ax.tile_extent) if cx[x] == 1 and wx[j, x] > 0]
            if ys and xs:
                src = to_storage(tiles[i][j], dtype)
                assert np.array_equal(gs[:, :, ys][:, :, :, xs],
                                      src[:, :, [y - oy for y in ys]][:, :, :, [x - ox for x in xs]])


@pytest.mark.parametrize("name", list(W.RAMP))
def test_full_workloads(tbl, name):
    w = W.RAMP[name]
    ay = tbl.RampAxis.spread(w.latent_hw[0], w.latent_tile, w.n_tiles[0], w.scale)
    ax = tbl.RampAxis.spread(w.latent_hw[1], w.latent_tile, w.n_tiles[1], w.scale)
    tiles = synth.smooth_field_tiles(w.seed, w.B, w.C, (ay.out_extent, ax.out_extent),
                                     [(o, ay.tile_extent) for o in ay.origins],
                                     [(o, ax.tile_extent) for o in ax.origins], w.dtype)
    _check(tbl, tiles, ay, ax, w.dtype)


LAYOUTS = [
    # (latent extent, latent tile, tiles, scale) per axis
    ((64, 32, 3, 8), (96, 32, 5, 8)),       # origins on 16-byte boundaries: 16-byte path
    ((40, 24, 3, 1), (77, 32, 4, 1)),       # latent space, odd origins: element path
    ((96, 32, 8, 1), (96, 32, 8, 8)),       # three tiles with weight at once
]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("layout", LAYOUTS, ids=["aligned", "odd", "dense"])
def test_small_layouts(tbl, dtype, layout):
    (ey, ty, ny, sy), (ex, tx, nx, sx) = layout
    ay = tbl.RampAxis.spread(ey, ty, ny, sy)
    ax = tbl.RampAxis.spread(ex, tx, nx, sx)
    rng = np.random.default_rng(len(dtype) + ny * nx)
    tiles = [[torch.from_numpy(rng.uniform(-1, 1, (2, 3, ay.tile_extent, ax.tile_extent))).to(TORCH[dtype])
              for _ in ax.origins] for _ in ay.origins]
    _check(tbl, tiles, ay, ax, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_tile_and_one_row_of_tiles(tbl, dtype):
    rng = np.random.default_rng(30)
    # a single tile is the canvas: copied exactly
    a1 = tbl.RampAxis.spread(32, 32, 1, 8)
    t = torch.from_numpy(rng.uniform(-1, 1, (2, 3, 256, 256))).to(TORCH[dtype])
    got = _run(tbl, [[t]], a1, a1, dtype)
    assert np.array_equal(to_storage(got, dtype), to_storage(t, dtype))
    # one row of tiles along the width: blends along x only
    ax = tbl.RampAxis.spread(96, 32, 4, 8)
    tiles = [[torch.from_numpy(rng.uniform(-1, 1, (1, 2, 256, ax.tile_extent))).to(TORCH[dtype])
              for _ in ax.origins]]
    _check(tbl, tiles, a1, ax, dtype)


def test_misaligned_pointers_take_the_element_path(tbl):
    ay = tbl.RampAxis.spread(64, 32, 3, 8)
    ax = tbl.RampAxis.spread(96, 32, 5, 8)
    rng = np.random.default_rng(31)
    shape = (1, 2, ay.tile_extent, ax.tile_extent)
    host = [[torch.from_numpy(rng.uniform(-1, 1, shape)).to(torch.bfloat16) for _ in ax.origins] for _ in ay.origins]
    keep, dev = [], []
    for row in host:
        drow = []
        for t in row:
            buf = torch.empty(t.numel() + 1, dtype=torch.bfloat16, device="cuda")
            v = buf[1:].view(shape)     # 2 bytes past a 16-byte boundary
            v.copy_(t)
            keep.append(buf)
            drow.append(v)
        dev.append(drow)
    out = torch.empty((1, 2, ay.out_extent, ax.out_extent), dtype=torch.bfloat16, device="cuda")
    tbl.tb_stitch2d_ramp(dev, ay, ax, out)
    torch.cuda.synchronize()
    exact = ramp_stitch_2d([[t.double().numpy() for t in row] for row in host], ay.origins, ax.origins,
                           ay.tile_extent, ax.tile_extent, (ay.out_extent, ax.out_extent), ay.zero, ay.ramp,
                           ax.zero, ax.ramp)
    assert violation(out.double().cpu().numpy(), exact, "bf16") <= 1.0


def test_empty_batch_and_guard_bands(tbl):
    ay = tbl.RampAxis.spread(64, 32, 3, 8)
    ax = tbl.RampAxis.spread(96, 32, 5, 8)
    empty = [[torch.empty((0, 3, ay.tile_extent, ax.tile_extent), device="cuda") for _ in ax.origins]
             for _ in ay.origins]
    tbl.tb_stitch2d_ramp(empty, ay, ax, torch.empty((0, 3, ay.out_extent, ax.out_extent), device="cuda"))
    # the output between two canary bands: nothing outside it is written
    rng = np.random.default_rng(32)
    tiles = [[torch.from_numpy(rng.uniform(-1, 1, (1, 3, ay.tile_extent, ax.tile_extent))).float().cuda()
              for _ in ax.origins] for _ in ay.origins]
    n = 3 * ay.out_extent * ax.out_extent
    guard = 4096
    buf = torch.full((n + 2 * guard,), 777.0, device="cuda")
    out = buf[guard:guard + n].view(1, 3, ay.out_extent, ax.out_extent)
    tbl.tb_stitch2d_ramp(tiles, ay, ax, out)
    torch.cuda.synchronize()
    assert (buf[:guard] == 777.0).all() and (buf[guard + n:] == 777.0).all()
    assert torch.isfinite(out).all()
