"""Normalised-ramp tile stitch, in float64 numpy.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: the page "Studio: size seam-free VAE tiles from measured peaks"
(unsloth PR #12764), commit "Decode this VAE in 32-latent tiles ...": tiles
of one size are spread over the canvas so the first starts at the edge and
the last ends at the opposite edge; a tile gets no weight within 4 latents of
an edge it shares with another tile, ramps to full weight over the next 8,
and the weights are normalised to 1 at every pixel.  The same page's encode
commit blends latent-space tiles the same way (scale 1).

Readings taken where the page gives words, not formulas:
  * the ramp is linear in the integer distance d (in samples) from the
    shared edge: r(d) = clamp((d - zero) / ramp, 0, 1), zero = 4 * scale,
    ramp = 8 * scale; the distance from the far edge of a tile of extent T at
    origin o is (o + T - 1) - p;
  * a tile's weight is the product of its ramps over its shared edges and
    over the axes (edges of the canvas are not shared and carry no ramp);
  * the output is sum(w * x) / sum(w) over the tiles covering the pixel,
    computed exactly (float64 here) and rounded once into the storage type.
"""
from typing import List, Sequence

import numpy as np


def axis_weights(origins: Sequence[int], extent: int, out_extent: int, zero: int, ramp: int) -> np.ndarray:
    """[N, out_extent] weight of tile n at each output position (0 outside
    the tile)."""
    n_t = len(origins)
    w = np.zeros((n_t, out_extent))
    for n, o in enumerate(origins):
        for q in range(extent):
            p = o + q
            if not (0 <= p < out_extent):
                continue
            r = 1.0
            if n > 0:                       # edge shared with tile n - 1
                r *= min(1.0, max(0.0, (q - zero) / ramp))
            if n < n_t - 1:                 # edge shared with tile n + 1
                r *= min(1.0, max(0.0, ((extent - 1 - q) - zero) / ramp))
            w[n, p] = r
    return w


def evenly_spread_origins(latent_extent: int, latent_tile: int, n_tiles: int, scale: int) -> List[int]:
    """Origins (output samples) of n_tiles tiles of latent_tile latents spread
    so the first starts at 0 and the last ends at the canvas edge: tile n at
    floor(n * (latent_extent - latent_tile) / (n_tiles - 1)) latents."""
    if n_tiles == 1:
        return [0]
    span = latent_extent - latent_tile
    return [(n * span // (n_tiles - 1)) * scale for n in range(n_tiles)]


def ramp_stitch_2d(tiles, origins_y, origins_x, extent_y: int, extent_x: int, out_hw, zero_y: int, ramp_y: int,
                   zero_x: int, ramp_x: int) -> np.ndarray:
    """float64 output [B, C, H, W] of the normalised-ramp stitch of
    ``tiles[i][j]`` ([B, C, extent_y, extent_x], any float dtype)."""
    H, W = out_hw
    wy = axis_weights(origins_y, extent_y, H, zero_y, ramp_y)
    wx = axis_weights(origins_x, extent_x, W, zero_x, ramp_x)
    B, C = np.asarray(tiles[0][0]).shape[:2]
    num = np.zeros((B, C, H, W))
    den = np.zeros((H, W))
    for i, oy in enumerate(origins_y):
        for j, ox in enumerate(origins_x):
            t = np.asarray(tiles[i][j], dtype=np.float64)
            w = np.outer(wy[i, oy:oy + extent_y], wx[j, ox:ox + extent_x])
            num[:, :, oy:oy + extent_y, ox:ox + extent_x] += t * w
            den[oy:oy + extent_y, ox:ox + extent_x] += w
    if (den <= 0).any():
        raise ValueError("a pixel has no tile with positive weight")
    return num / den
