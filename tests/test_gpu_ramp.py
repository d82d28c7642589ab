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
        ref = R.storage_to_f64(R.round_f64(exact, dtype), dtype)
        mant = 10 if dtype == "f16" else 7
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -8))) - mant)
        assert (np.abs(g - ref) <= ulp).all()
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
