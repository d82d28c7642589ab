"""Pins for the normalised-ramp stitch oracle (oracle/ramp.py): a closed-form
cross-fade, invariances of a normalised weighted average, and degenerate
layouts with a known answer."""
import numpy as np
import pytest

from oracle.ramp import axis_weights, evenly_spread_origins, ramp_stitch_2d


def _tiles(rng, oy, ox, ey, ex, B=1, C=2):
    return [[rng.standard_normal((B, C, ey, ex)) for _ in ox] for _ in oy]


def test_weights_follow_the_stated_ramp():
    # zero weight within 4 latents of a shared edge, full weight 8 latents later
    s = 2
    w = axis_weights([0, 40], 64, 104, 4 * s, 8 * s)
    q = np.arange(64)
    left_of_tile1 = w[1, 40 + q]
    assert (left_of_tile1[:8] == 0).all()
    assert left_of_tile1[8 + 16:64 - 24].min() == 1.0
    assert np.allclose(left_of_tile1[8:24], np.arange(16) / 16)
    # canvas edges carry no ramp
    assert w[0, 0] == 1.0 and w[1, 103] == 1.0


def test_every_pixel_has_positive_total_weight_with_16_latent_overlaps():
    for ext, tile in ((64, 32), (100, 32), (256, 32), (77, 40)):
        n = 1
        while n == 1 or (tile - (ext - tile) // (n - 1)) < 16:
            n += 1
        org = evenly_spread_origins(ext, tile, n, 8)
        w = axis_weights(org, tile * 8, ext * 8, 32, 64)
        assert org[0] == 0 and org[-1] + tile * 8 == ext * 8
        assert (w.sum(axis=0) > 0).all()


def test_crossfade_closed_form_when_the_ramps_meet():
    # overlap of exactly zero + ramp + zero + 1 samples: the two ramps are
    # complementary, so the stitch is the plain linear cross-fade
    zero, ramp, ext = 3, 10, 40
    ov = 2 * zero + ramp + 1
    org = [0, ext - ov]
    W = org[1] + ext
    rng = np.random.default_rng(1)
    tiles = _tiles(rng, [0], org, 4, ext)
    out = ramp_stitch_2d(tiles, [0], org, 4, ext, (4, W), 0, 1, zero, ramp)
    a, b = tiles[0][0], tiles[0][1]
    for p in range(W):
        if p < org[1] + zero:
            ref = a[..., p]
        elif p >= org[1] + zero + ramp:
            ref = b[..., p - org[1]]
        else:
            wb = (p - org[1] - zero) / ramp
            ref = (1 - wb) * a[..., p] + wb * b[..., p - org[1]]
        assert np.abs(out[..., p] - ref).max() < 1e-13


def test_constant_and_affine_invariance():
    rng = np.random.default_rng(2)
    oy = evenly_spread_origins(60, 32, 3, 2)
    ox = evenly_spread_origins(90, 32, 5, 2)
    ey, ex = 64, 64
    H, W = 120, 180
    const = [[np.full((1, 1, ey, ex), 0.3) for _ in ox] for _ in oy]
    out = ramp_stitch_2d(const, oy, ox, ey, ex, (H, W), 8, 16, 8, 16)
    assert np.abs(out - 0.3).max() < 1e-15
    t = _tiles(rng, oy, ox, ey, ex)
    base = ramp_stitch_2d(t, oy, ox, ey, ex, (H, W), 8, 16, 8, 16)
    t2 = [[2.5 * x - 1.0 for x in row] for row in t]
    aff = ramp_stitch_2d(t2, oy, ox, ey, ex, (H, W), 8, 16, 8, 16)
    assert np.abs(aff - (2.5 * base - 1.0)).max() < 1e-12


def test_single_tile_is_the_tile_and_unshared_interior_is_copied():
    rng = np.random.default_rng(3)
    t = _tiles(rng, [0], [0], 16, 24)
    out = ramp_stitch_2d(t, [0], [0], 16, 24, (16, 24), 4, 8, 4, 8)
    assert np.array_equal(out, t[0][0])
    # a 1x2 grid: pixels of tile 0 before tile 1 starts are tile 0 exactly
    t = _tiles(rng, [0], [0, 20], 8, 40)
    out = ramp_stitch_2d(t, [0], [0, 20], 8, 40, (8, 60), 0, 1, 4, 8)
    assert np.array_equal(out[..., :20], t[0][0][..., :20])
    assert np.array_equal(out[..., 40:], t[0][1][..., 20:])


def test_a_pixel_without_weight_is_refused():
    with pytest.raises(ValueError):
        # overlap too short for the zero bands: the seam has no weight
        t = _tiles(np.random.default_rng(4), [0], [0, 30], 4, 36)
        ramp_stitch_2d(t, [0], [0, 30], 4, 36, (4, 66), 0, 1, 4, 8)


def test_spread_is_even_edge_to_edge_and_covering():
    # what the page fixes about the spread: the first tile at 0, the last
    # ending at the edge, and the tiles equally spaced -- in whole latents the
    # gaps can differ by one at most -- with no sample left uncovered
    import random
    rnd = random.Random(17)
    for _ in range(400):
        tile = rnd.randint(4, 96)
        ext = rnd.randint(tile, 12 * tile)
        lo = 1 if ext == tile else 2
        n = rnd.randint(lo, lo + 10)
        if n == 1:
            continue
        scale = rnd.choice([1, 8, 16])
        org = evenly_spread_origins(ext, tile, n, scale)
        lat = [o // scale for o in org]
        assert all(o % scale == 0 for o in org)
        assert lat[0] == 0 and lat[-1] + tile == ext
        gaps = [b - a for a, b in zip(lat, lat[1:])]
        assert max(gaps) - min(gaps) <= 1
        assert sum(gaps) == ext - tile
        # the spread never runs ahead of the exact equal spacing
        assert all(l * (n - 1) <= k * (ext - tile) for k, l in enumerate(lat))
