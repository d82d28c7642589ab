"""Named synthetic workloads: tile-grid parameters, shapes and input recipe.

Each stitch workload is a decoded image or clip cut into overlapping tiles by
the stock tiled-decode rule (latent tile, overlap factor, latent scale); the
tiles are drawn by ``synth``.  The PatchGroupNorm workloads are decoder
activations split into four patches along one spatial axis; the Patchify
workloads split such activations among ranks and gather them back.

The generator needs each tile's placement (output-space origin, extent);
callers pass it from a derived geometry -- ``tileblend.tb_axis_layout`` in
the product path, the oracle's geometry in the tests.
"""
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

from . import synth


@dataclass(frozen=True)
class AxisSpec:
    latent_extent: int
    latent_tile: int
    overlap: float
    scale: int


@dataclass(frozen=True)
class StitchWorkload:
    name: str
    dtype: str                 # 'f32' | 'f16' | 'bf16'
    B: int
    C: int
    axes: Tuple[AxisSpec, ...]  # (y, x) or (t, y, x)
    recipe: str                # 'smooth' | 'uniform' | 'spacetime'
    seed: int

    @property
    def ndim(self) -> int:
        return len(self.axes)


def _img(extent_lat, tile=64, ov=0.25, scale=8):
    return AxisSpec(extent_lat, tile, ov, scale)


STITCH = {
    # 2D, fp32, 1024x1024, 3x3 grid of 512 px tiles (blend 128, row_limit 384)
    "image_1024_f32": StitchWorkload("image_1024_f32", "f32", 1, 3, (_img(128), _img(128)), "smooth", 1234),
    # 2D, batch 4, 2048x2048, 6x6 grid, last tiles 128 px
    "image_2048_f16": StitchWorkload("image_2048_f16", "f16", 4, 3, (_img(256), _img(256)), "smooth", 1235),
    "image_2048_bf16": StitchWorkload("image_2048_bf16", "bf16", 4, 3, (_img(256), _img(256)), "smooth", 1235),
    "image_2048_f16_uniform": StitchWorkload("image_2048_f16_uniform", "f16", 4, 3, (_img(256), _img(256)),
                                             "uniform", 1335),
    "image_2048_bf16_uniform": StitchWorkload("image_2048_bf16_uniform", "bf16", 4, 3, (_img(256), _img(256)),
                                              "uniform", 1335),
    # 2D, 1600x2048 (latent 200x256), 120x72-latent tiles: per-axis blends, clamped slivers
    "wide_1600x2048_bf16": StitchWorkload("wide_1600x2048_bf16", "bf16", 1, 3, (_img(200, 120), _img(256, 72)),
                                          "smooth", 1236),
    # 3D, 49 frames of 480x832: 16-frame tiles (stride 12, blend 4), 256 px tiles (stride 192, blend 64)
    "video_49x480x832_bf16": StitchWorkload("video_49x480x832_bf16", "bf16", 1, 3,
                                            (AxisSpec(49, 16, 0.25, 1), _img(60, 32), _img(104, 32)),
                                            "spacetime", 1237),
}


@dataclass(frozen=True)
class RampWorkload:
    """Equally sized tiles spread over the canvas (first at 0, last at the
    edge), blended with the normalised ramp: zero weight for 4 latents next
    to a shared edge, full weight 8 latents later."""
    name: str
    dtype: str
    B: int
    C: int
    latent_hw: Tuple[int, int]
    latent_tile: int
    n_tiles: Tuple[int, int]
    scale: int
    recipe: str
    seed: int


RAMP = {
    # decoded tiles: 2048x2048 (256 latents at 8x), 64-latent tiles, 16-latent overlaps
    "ramp_2048_bf16": RampWorkload("ramp_2048_bf16", "bf16", 1, 3, (256, 256), 64, (5, 5), 8, "smooth", 1240),
    # latent-space tiles of a tiled encode: batch 4, 16 channels, 256x256 latents (a 2048 px image at 8x),
    # 64-latent tiles with 32-latent overlaps
    "ramp_latent_256_bf16": RampWorkload("ramp_latent_256_bf16", "bf16", 4, 16, (256, 256), 64, (7, 7), 1,
                                         "smooth", 1241),
}


@dataclass(frozen=True)
class GroupNormWorkload:
    name: str
    dtype: str
    shape: Tuple[int, ...]     # unsharded [N, C, *spatial]
    split_dim: int
    patches: int
    patch_means: Tuple[float, ...]
    groups: int
    eps: float
    seed: int


GROUPNORM = {
    "gn_4d_1x512x256x256": GroupNormWorkload("gn_4d_1x512x256x256", "bf16", (1, 512, 256, 256), 2, 4,
                                             (-3.0, -1.0, 1.0, 3.0), 32, 1e-6, 1238),
    "gn_5d_1x384x13x120x208": GroupNormWorkload("gn_5d_1x384x13x120x208", "bf16", (1, 384, 13, 120, 208), 4, 4,
                                                (-3.0, -1.0, 1.0, 3.0), 32, 1e-6, 1239),
}


@dataclass(frozen=True)
class PatchifyWorkload:
    """An activation split among ranks along one axis in whole bands of
    ``factor`` positions (the first ranks one band more), and gathered back."""
    name: str
    dtype: str
    shape: Tuple[int, ...]
    axis: int
    factor: int
    ranks: int
    seed: int


PATCHIFY = {
    # the 4D decoder activation of the GroupNorm workload, 4 ranks along the height: 64 rows each
    "patchify_4d_1x512x256x256_h4": PatchifyWorkload("patchify_4d_1x512x256x256_h4", "bf16", (1, 512, 256, 256),
                                                     2, 8, 4, 1242),
    # the 5D activation, 3 ranks along the width: 26 bands of 8 -> 72, 72, 64 columns
    "patchify_5d_1x384x13x120x208_w3": PatchifyWorkload("patchify_5d_1x384x13x120x208_w3", "bf16",
                                                        (1, 384, 13, 120, 208), 4, 8, 3, 1243),
}


def make_stitch_tiles(w: StitchWorkload, boxes: Sequence[Sequence[Tuple[int, int]]], out_extents: Sequence[int]):
    """CPU tiles of workload ``w``; ``boxes[a]`` lists (origin, extent) of the
    tiles along axis a and ``out_extents`` the output extents."""
    bx = boxes
    if w.ndim == 2:
        if w.recipe == "uniform":
            return synth.uniform_tiles(w.seed, w.B, w.C, bx[0], bx[1], w.dtype)
        return synth.smooth_field_tiles(w.seed, w.B, w.C, tuple(out_extents), bx[0], bx[1], w.dtype)
    return synth.spacetime_field_tiles(w.seed, w.B, w.C, tuple(out_extents), bx[0], bx[1], bx[2], w.dtype)


def make_groupnorm_inputs(w: GroupNormWorkload):
    return synth.groupnorm_patches(w.seed, w.shape, w.split_dim, w.patches, w.patch_means, w.dtype)


def make_ramp_tiles(w: RampWorkload, ay, ax):
    """CPU tiles of a ramp workload cut from one smooth field; ``ay`` / ``ax``
    carry the tile origins and extents (samples)."""
    return synth.smooth_field_tiles(w.seed, w.B, w.C, (ay.out_extent, ax.out_extent),
                                    [(o, ay.tile_extent) for o in ay.origins],
                                    [(o, ax.tile_extent) for o in ax.origins], w.dtype)


def make_patchify_input(w: PatchifyWorkload):
    return synth.normal_tensor(w.seed, w.shape, w.dtype)
