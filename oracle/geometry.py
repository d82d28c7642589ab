"""Stock tiled-decode grid geometry, in plain Python.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages name the geometry's parameters -- latent tile size, overlap factor,
scale factor, blend_extent and row_limit -- and show their stock relation in
pixels on the page "Studio: size seam-free VAE tiles from measured peaks"
(unsloth PR #12764, commit "Decode this VAE in 32-latent tiles ...": a
16-latent tile at 16x is 256 px with a 192 px stride and a 64 px blend).
Their plainest reading, the one the tiled decode in diffusers uses, is:

    stride        = int(latent_tile * (1 - overlap))            (latents)
    tile origins  = range(0, latent_extent, stride)              (latents)
    tile extent   = min(latent_tile, latent_extent - origin) * scale   (px)
    blend_extent  = int(latent_tile * scale * overlap)           (px)
    row_limit     = latent_tile * scale - blend_extent           (px)

Per pair of neighbouring tiles the blend extent is clamped to what both
tiles hold (page "[Proposal] Vectorize tiled VAE blending ...", "Proposed
scope", which keeps that clamp when vectorising):

    e(n) = min(extent(n-1), extent(n), blend_extent),   e(0) = 0

and each tile keeps its first min(extent, row_limit) slices, which are then
concatenated, so the output extent is the sum of the kept extents.
"""
from dataclasses import dataclass
from typing import List, Optional


@dataclass(frozen=True)
class AxisLayout:
    stride: int            # latents between tile origins
    origins: List[int]     # tile origins, latents
    extents: List[int]     # decoded tile extents, px (or frames)
    blend_extent: int      # px
    row_limit: int         # px
    blends: List[int]      # clamped blend extent e(n) against tile n-1; e(0) = 0
    kept: List[int]        # min(extent, row_limit)
    offsets: List[int]     # output offset of each tile's kept part
    out_extent: int        # sum of kept

    @property
    def n(self) -> int:
        return len(self.extents)


def axis_layout(latent_extent: int, latent_tile: int, overlap: float, scale: int,
                blend_extent: Optional[int] = None, row_limit: Optional[int] = None) -> AxisLayout:
    """Geometry of one axis of the tile grid.

    ``blend_extent`` / ``row_limit`` of ``None`` take the stock values
    derived from the tile size and overlap factor.
    """
    stride = int(latent_tile * (1 - overlap))
    if stride <= 0:
        raise ValueError("overlap leaves no stride between tiles")
    if blend_extent is None:
        blend_extent = int(latent_tile * scale * overlap)
    if row_limit is None:
        row_limit = latent_tile * scale - blend_extent
    origins = list(range(0, latent_extent, stride))
    extents = [min(latent_tile, latent_extent - o) * scale for o in origins]
    blends = [0 if n == 0 else min(extents[n - 1], extents[n], blend_extent) for n in range(len(extents))]
    kept = [min(L, row_limit) for L in extents]
    offsets = []
    acc = 0
    for k in kept:
        offsets.append(acc)
        acc += k
    return AxisLayout(stride, origins, extents, blend_extent, row_limit, blends, kept, offsets, acc)


def single_axis(extent: int) -> AxisLayout:
    """A degenerate axis holding one tile of ``extent`` and no blending
    (used for the frame axis of a 2D image)."""
    return AxisLayout(extent, [0], [extent], 0, extent, [0], [extent], [0], extent)
