"""Pins for the oracle's stitch (oracle/stitch.c) that do not come from the
oracle itself: degenerate cases with a known answer, the algebraic closed
form of the recurrence (float64 storage mode), and a brute-force replay of
the blend loops in torch CPU arithmetic on tiny grids."""
import itertools

import numpy as np
import pytest
import torch

from oracle.geometry import axis_layout, single_axis
from oracle.stitch import stitch
from oracle import rounding as R
from patch_groupnorm_gb300 import synth
from tests.stitch_helpers import TORCH, boxes, from_storage, to_storage, torch_replay_2d, torch_replay_3d

NARROW = ["f32", "f16", "bf16"]


def _random_tiles_2d(rng, B, C, ay, ax, dtype):
    return [[torch.from_numpy(rng.uniform(-1, 1, (B, C, ly, lx))).to(TORCH[dtype])
             for lx in ax.extents] for ly in ay.extents]


def _storage_grid(tiles, dtype):
    if isinstance(tiles, torch.Tensor):
        return to_storage(tiles, dtype)
    return [_storage_grid(t, dtype) for t in tiles]


# --------------------------------------------------------------------------
# degenerate cases with a known answer
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", NARROW)
def test_zero_overlap_is_concat_of_crops(dtype):
    rng = np.random.default_rng(10)
    ay = axis_layout(30, 8, 0.0, 4)          # extents 32,32,32,24; no blend
    ax = axis_layout(21, 8, 0.0, 4, row_limit=24)  # crop below the extent
    assert all(e == 0 for e in ay.blends + ax.blends)
    tiles = _random_tiles_2d(rng, 2, 3, ay, ax, dtype)
    out = stitch(_storage_grid(tiles, dtype), (ay, ax), dtype)
    ref = torch.cat([torch.cat([t[..., :ay.row_limit, :ax.row_limit] for t in row], -1) for row in tiles], -2)
    assert np.array_equal(out, to_storage(ref, dtype))


@pytest.mark.parametrize("dtype", NARROW)
def test_single_tile_grid_is_the_tile(dtype):
    rng = np.random.default_rng(11)
    ay = axis_layout(20, 64, 0.25, 8)
    ax = axis_layout(33, 64, 0.25, 8)
    assert ay.n == 1 and ax.n == 1
    tiles = _random_tiles_2d(rng, 1, 3, ay, ax, dtype)
    out = stitch(_storage_grid(tiles, dtype), (ay, ax), dtype)
    assert np.array_equal(out, to_storage(tiles[0][0], dtype))


@pytest.mark.parametrize("dtype", NARROW)
def test_constant_zero_tiles_stay_zero(dtype):
    ay = axis_layout(20, 8, 0.25, 4)
    ax = axis_layout(17, 8, 0.5, 4)
    tiles = [[torch.zeros(1, 2, ly, lx, dtype=TORCH[dtype]) for lx in ax.extents] for ly in ay.extents]
    out = stitch(_storage_grid(tiles, dtype), (ay, ax), dtype)
    assert (R.storage_to_f64(out, dtype) == 0).all()


def test_constant_tiles_exact_when_every_operation_is_exact():
    # fp32, power-of-two blend extents and a value with few significant bits:
    # every coefficient c/e is a dyadic rational, every product and sum exact.
    ay = axis_layout(24, 8, 0.25, 8)   # blend 16
    ax = axis_layout(40, 16, 0.25, 2)  # blend 8
    assert ay.blend_extent == 16 and ax.blend_extent == 8
    tiles = [[torch.full((1, 1, ly, lx), 0.375) for lx in ax.extents] for ly in ay.extents]
    out = stitch(_storage_grid(tiles, "f32"), (ay, ax), "f32")
    assert (out == np.float32(0.375)).all()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_constant_tiles_stay_within_one_ulp(dtype):
    ay = axis_layout(40, 16, 0.25, 8)   # blend 32, 3 tiles
    ax = axis_layout(50, 24, 0.25, 6)   # blend 36
    c = torch.tensor(0.7, dtype=TORCH[dtype])
    tiles = [[torch.full((1, 1, ly, lx), float(c), dtype=TORCH[dtype]) for lx in ax.extents] for ly in ay.extents]
    out = R.storage_to_f64(stitch(_storage_grid(tiles, dtype), (ay, ax), dtype), dtype)
    ulp = 2.0 ** (-10 if dtype == "f16" else -7) * 0.5  # spacing just below 1
    assert np.abs(out - float(c)).max() <= ulp


# --------------------------------------------------------------------------
# closed form of the recurrence (float64 storage: no narrowing, double
# coefficients), derived by hand:
#   band along one axis:      (1 - w) a + w b
#   corner, axes blended in the order first (w1) then second (w2):
#     D (1-w2)(1-w1)(1+w2) + L (1-w2) w1 + A w2^2 (1-w1) + T w2 w1
#   with T the tile itself, A its neighbour along the first axis, L along the
#   second, D the diagonal one; the four weights sum to 1.
# --------------------------------------------------------------------------

def _corner(D, A, L, T, w1, w2):
    return D * (1 - w2) * (1 - w1) * (1 + w2) + L * (1 - w2) * w1 + A * w2 * w2 * (1 - w1) + T * w2 * w1


def test_corner_weights_sum_to_one():
    for w1, w2 in itertools.product(np.linspace(0, 1, 7), repeat=2):
        assert abs(_corner(1.0, 1.0, 1.0, 1.0, w1, w2) - 1.0) < 1e-15


def test_closed_form_2x2_grid_float64():
    rng = np.random.default_rng(12)
    ay = axis_layout(12, 8, 0.25, 2)    # extents 16, 12 px -> e_y = 4
    ax = axis_layout(6, 6, 0.5, 3)      # extents 18, 9 px  -> e_x = 9 (whole second tile)
    assert ay.n == 2 and ax.n == 2
    R_ = [[rng.standard_normal((2, 1, ly, lx)) for lx in ax.extents] for ly in ay.extents]
    out = stitch(R_, (ay, ax), "f64")
    ey, ex = ay.blends[1], ax.blends[1]
    Ly0, Lx0 = ay.extents[0], ax.extents[0]
    ref = np.zeros_like(out)
    for i, j in itertools.product(range(2), range(2)):
        for cy in range(ay.kept[i]):
            for cx in range(ax.kept[j]):
                oy, ox = ay.offsets[i] + cy, ax.offsets[j] + cx
                T = R_[i][j][..., cy, cx]
                in_y = i == 1 and cy < ey
                in_x = j == 1 and cx < ex
                wy, wx = (cy / ey if in_y else 0.0), (cx / ex if in_x else 0.0)
                if in_y and in_x:
                    D = R_[0][0][..., Ly0 - ey + cy, Lx0 - ex + cx]
                    A = R_[0][1][..., Ly0 - ey + cy, cx]
                    L = R_[1][0][..., cy, Lx0 - ex + cx]
                    v = _corner(D, A, L, T, wy, wx)
                elif in_y:
                    v = (1 - wy) * R_[0][j][..., Ly0 - ey + cy, cx] + wy * T
                elif in_x:
                    v = (1 - wx) * R_[i][0][..., cy, Lx0 - ex + cx] + wx * T
                else:
                    v = T
                ref[..., oy, ox] = v
    assert np.abs(out - ref).max() < 1e-13


def test_closed_form_chain_of_three_tiles_float64():
    # a middle tile both receives a band (at its top) and lends one (from its
    # bottom); with the bands apart, the lent rows are its raw rows.
    rng = np.random.default_rng(13)
    ay = axis_layout(22, 8, 0.25, 4)    # stride 6: extents 32, 32, 32, 16 px
    ax = single_axis(5)
    R_ = [[rng.standard_normal((1, 2, L, 5))] for L in ay.extents]
    out = stitch(R_, (ay, ax), "f64")
    ref = np.zeros_like(out)
    for i in range(ay.n):
        e = ay.blends[i]
        for cy in range(ay.kept[i]):
            T = R_[i][0][..., cy, :]
            if i > 0 and cy < e:
                assert ay.extents[i - 1] - e + cy >= ay.blends[i - 1]  # lent rows are unblended
                v = (1 - cy / e) * R_[i - 1][0][..., ay.extents[i - 1] - e + cy, :] + (cy / e) * T
            else:
                v = T
            ref[..., ay.offsets[i] + cy, :] = v
    assert np.abs(out - ref).max() < 1e-13


def test_closed_form_time_then_height_corner_float64():
    rng = np.random.default_rng(14)
    at = axis_layout(6, 5, 0.4, 1)      # frames: extents 5, 3 (stride 3), e_t = 2
    ay = axis_layout(5, 4, 0.25, 2)     # extents 8, 4 (stride 3), e_y = 2
    ax = single_axis(3)
    assert at.n == 2 and ay.n == 2
    R_ = [[[rng.standard_normal((1, 1, lt, ly, 3))] for ly in ay.extents] for lt in at.extents]
    out = stitch(R_, (at, ay, ax), "f64")
    et, ey = at.blends[1], ay.blends[1]
    Lt0, Ly0 = at.extents[0], ay.extents[0]
    k, i = 1, 1
    for ct in range(min(et, at.kept[1])):
        for cy in range(min(ey, ay.kept[1])):
            wt, wy = ct / et, cy / ey
            D = R_[0][0][0][..., Lt0 - et + ct, Ly0 - ey + cy, :]
            A = R_[0][1][0][..., Lt0 - et + ct, cy, :]      # neighbour along time
            L = R_[1][0][0][..., ct, Ly0 - ey + cy, :]      # neighbour along height
            T = R_[1][1][0][..., ct, cy, :]
            ref = _corner(D, A, L, T, wt, wy)
            got = out[..., at.offsets[k] + ct, ay.offsets[i] + cy, :]
            assert np.abs(got - ref).max() < 1e-13


@pytest.mark.parametrize("dtype", NARROW)
def test_3d_with_one_frame_tile_equals_2d_per_frame(dtype):
    rng = np.random.default_rng(15)
    ay = axis_layout(11, 6, 0.5, 2)
    ax = axis_layout(9, 4, 0.25, 3)
    at = single_axis(3)
    tiles3 = [[[torch.from_numpy(rng.uniform(-1, 1, (1, 2, 3, ly, lx))).to(TORCH[dtype])
                for lx in ax.extents] for ly in ay.extents]]
    out3 = stitch(_storage_grid(tiles3, dtype), (at, ay, ax), dtype)
    for f in range(3):
        tiles2 = [[t[:, :, f].contiguous() for t in row] for row in tiles3[0]]
        out2 = stitch(_storage_grid(tiles2, dtype), (ay, ax), dtype)
        assert np.array_equal(out3[:, :, f], out2)


# --------------------------------------------------------------------------
# brute-force replay of the blend loops in torch CPU arithmetic
# --------------------------------------------------------------------------

GEOMS_2D = [
    # (latent extent, latent tile, overlap, scale) per axis
    ((20, 8, 0.25, 4), (26, 8, 0.25, 4)),
    ((17, 6, 0.5, 3), (9, 5, 0.2, 5)),      # half overlap, odd extents
    ((31, 12, 0.25, 2), (13, 4, 0.25, 8)),  # slivers of 1 and 2 latents
    ((10, 4, 0.75, 4), (10, 4, 0.6, 4)),    # bands that chain (overlap > 1/2)
]


@pytest.mark.parametrize("dtype", NARROW)
@pytest.mark.parametrize("geom", GEOMS_2D, ids=lambda g: "x".join(str(a[0]) for a in g))
def test_oracle_matches_torch_replay_2d(dtype, geom):
    rng = np.random.default_rng(hash(geom) % 2 ** 32)
    ay, ax = (axis_layout(*a) for a in geom)
    tiles = _random_tiles_2d(rng, 2, 2, ay, ax, dtype)
    out = stitch(_storage_grid(tiles, dtype), (ay, ax), dtype)
    ref = torch_replay_2d(tiles, ay.blend_extent, ay.row_limit, ax.blend_extent, ax.row_limit)
    assert np.array_equal(out, to_storage(ref, dtype))


@pytest.mark.parametrize("dtype", NARROW)
def test_oracle_matches_torch_replay_3d(dtype):
    rng = np.random.default_rng(16)
    at = axis_layout(13, 5, 0.25, 1)        # frames 5,5,5,1 -> e_t 1,1,1
    ay = axis_layout(7, 4, 0.5, 2)
    ax = axis_layout(9, 4, 0.25, 3)
    tiles = [[[torch.from_numpy(rng.uniform(-1, 1, (1, 2, lt, ly, lx))).to(TORCH[dtype])
               for lx in ax.extents] for ly in ay.extents] for lt in at.extents]
    out = stitch(_storage_grid(tiles, dtype), (at, ay, ax), dtype)
    ref = torch_replay_3d(tiles, at.blend_extent, at.row_limit, ay.blend_extent, ay.row_limit,
                          ax.blend_extent, ax.row_limit)
    assert np.array_equal(out, to_storage(ref, dtype))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_oracle_matches_torch_replay_on_smooth_field(dtype):
    # the synthetic smooth field at a small size, the recipe the workloads use
    ay = axis_layout(32, 16, 0.25, 4)
    ax = axis_layout(40, 16, 0.25, 4)
    tiles = synth.smooth_field_tiles(7, 1, 3, (ay.out_extent, ax.out_extent), boxes(ay, 4), boxes(ax, 4), dtype)
    out = stitch(_storage_grid(tiles, dtype), (ay, ax), dtype)
    ref = torch_replay_2d(tiles, ay.blend_extent, ay.row_limit, ax.blend_extent, ax.row_limit)
    assert np.array_equal(out, to_storage(ref, dtype))
