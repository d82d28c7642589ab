"""Seeded synthetic inputs for the stitch and PatchGroupNorm.

This module draws numbers only: it holds none of the method's arithmetic (no
tile geometry, no blending, no normalisation).  The caller passes each tile's
placement -- its output-space origin and extent per axis -- and gets back
tensors on the CPU, generated in float64 and cast with torch's
round-to-nearest-even.  Both the CUDA path and the oracle are fed from here.

Recipes (decoded VAE tiles and decoder activations stand in for real ones):

* smooth field: per (batch, channel) a sum of ``n_waves`` 2D sinusoids of
  amplitude ``amp / n_waves`` each, frequencies U(0.5, 6) cycles per image,
  phases U(0, 2 pi); each tile is the field over its own footprint plus a
  per-(tile, batch, channel) offset U(-0.1, 0.1) and i.i.d. N(0, 0.05^2).
* uniform: i.i.d. U(-1, 1) per tile element (rounding stress).
* space-time field: as the smooth field with ``n_waves`` sinusoids in
  (t, y, x), temporal frequency U(0.5, 4) cycles per clip.
* GroupNorm patches: patch p ~ N(mu_p, 1), gamma ~ N(1, 0.1^2),
  beta ~ N(0, 0.1^2).
* activation: one tensor of i.i.d. N(0, 1) (the input of a patch split).
"""
import math
from typing import List, Sequence, Tuple

import torch

Box = Tuple[int, int]  # (origin in output space, extent)

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "f64": torch.float64}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def _uniform(g: torch.Generator, shape, lo: float, hi: float) -> torch.Tensor:
    return torch.rand(shape, generator=g, dtype=torch.float64) * (hi - lo) + lo


def smooth_field_tiles(seed: int, B: int, C: int, out_hw: Tuple[int, int], boxes_y: Sequence[Box],
                       boxes_x: Sequence[Box], dtype: str, n_waves: int = 8, amp: float = 0.8,
                       offset: float = 0.1, noise: float = 0.05) -> List[List[torch.Tensor]]:
    """Tiles[i][j] of shape [B, C, extent_y(i), extent_x(j)] cut from one
    seeded smooth field over an ``out_hw`` image."""
    g = _gen(seed)
    H, W = out_hw
    fy = _uniform(g, (B, C, n_waves), 0.5, 6.0)
    fx = _uniform(g, (B, C, n_waves), 0.5, 6.0)
    ph = _uniform(g, (B, C, n_waves), 0.0, 2 * math.pi)
    a = amp / n_waves
    tiles = []
    for (oy, ly) in boxes_y:
        row = []
        y = torch.arange(oy, oy + ly, dtype=torch.float64)
        for (ox, lx) in boxes_x:
            x = torch.arange(ox, ox + lx, dtype=torch.float64)
            # sin(p + q) = sin p cos q + cos p sin q, evaluated as outer products
            py = 2 * math.pi * fy[..., None] * (y / H) + ph[..., None]      # [B, C, K, ly]
            qx = 2 * math.pi * fx[..., None] * (x / W)                      # [B, C, K, lx]
            f = a * (torch.einsum("bcky,bckx->bcyx", torch.sin(py), torch.cos(qx))
                     + torch.einsum("bcky,bckx->bcyx", torch.cos(py), torch.sin(qx)))
            f = f + _uniform(g, (B, C, 1, 1), -offset, offset)
            f = f + noise * torch.randn((B, C, ly, lx), generator=g, dtype=torch.float64)
            row.append(f.to(TORCH_DTYPES[dtype]).contiguous())
        tiles.append(row)
    return tiles


def uniform_tiles(seed: int, B: int, C: int, boxes_y: Sequence[Box], boxes_x: Sequence[Box],
                  dtype: str) -> List[List[torch.Tensor]]:
    """Tiles[i][j] of i.i.d. U(-1, 1) values."""
    g = _gen(seed)
    return [[_uniform(g, (B, C, ly, lx), -1.0, 1.0).to(TORCH_DTYPES[dtype]).contiguous()
             for (_, lx) in boxes_x] for (_, ly) in boxes_y]


def spacetime_field_tiles(seed: int, B: int, C: int, out_thw: Tuple[int, int, int], boxes_t: Sequence[Box],
                          boxes_y: Sequence[Box], boxes_x: Sequence[Box], dtype: str, n_waves: int = 16,
                          amp: float = 0.8, offset: float = 0.1, noise: float = 0.05) -> List[List[List[torch.Tensor]]]:
    """Tiles[k][i][j] of shape [B, C, extent_t(k), extent_y(i), extent_x(j)]
    cut from one seeded space-time field over a ``out_thw`` clip."""
    g = _gen(seed)
    T, H, W = out_thw
    ft = _uniform(g, (B, C, n_waves), 0.5, 4.0)
    fy = _uniform(g, (B, C, n_waves), 0.5, 6.0)
    fx = _uniform(g, (B, C, n_waves), 0.5, 6.0)
    ph = _uniform(g, (B, C, n_waves), 0.0, 2 * math.pi)
    a = amp / n_waves
    out = []
    for (ot, lt) in boxes_t:
        t = torch.arange(ot, ot + lt, dtype=torch.float64)
        plane = []
        for (oy, ly) in boxes_y:
            y = torch.arange(oy, oy + ly, dtype=torch.float64)
            row = []
            for (ox, lx) in boxes_x:
                x = torch.arange(ox, ox + lx, dtype=torch.float64)
                pt = 2 * math.pi * ft[..., None] * (t / T) + ph[..., None]   # [B,C,K,lt]
                py = 2 * math.pi * fy[..., None] * (y / H)                    # [B,C,K,ly]
                qx = 2 * math.pi * fx[..., None] * (x / W)                    # [B,C,K,lx]
                # phase p(t) + q(y) + r(x): expand sin of the sum into products
                st, ct = torch.sin(pt), torch.cos(pt)
                sy, cy = torch.sin(py), torch.cos(py)
                sx, cx = torch.sin(qx), torch.cos(qx)
                # sin(a+b) = sa*cb + ca*sb with a = t + y, b = x
                sa = torch.einsum("bckt,bcky->bckty", st, cy) + torch.einsum("bckt,bcky->bckty", ct, sy)
                ca = torch.einsum("bckt,bcky->bckty", ct, cy) - torch.einsum("bckt,bcky->bckty", st, sy)
                f = a * (torch.einsum("bckty,bckx->bctyx", sa, cx) + torch.einsum("bckty,bckx->bctyx", ca, sx))
                f = f + _uniform(g, (B, C, 1, 1, 1), -offset, offset)
                f = f + noise * torch.randn((B, C, lt, ly, lx), generator=g, dtype=torch.float64)
                row.append(f.to(TORCH_DTYPES[dtype]).contiguous())
            plane.append(row)
        out.append(plane)
    return out


def groupnorm_patches(seed: int, full_shape: Sequence[int], split_dim: int, n_patches: int,
                      patch_means: Sequence[float], dtype: str):
    """Split a [N, C, *spatial] activation into ``n_patches`` contiguous
    patches along ``split_dim`` (a spatial dim, >= 2); patch p is drawn from
    N(patch_means[p], 1).  Also returns gamma ~ N(1, 0.1^2) and
    beta ~ N(0, 0.1^2) of shape [C].  Sizes along the split dim differ by at
    most one (the first patches take the remainder)."""
    g = _gen(seed)
    full_shape = list(full_shape)
    size = full_shape[split_dim]
    base, rem = divmod(size, n_patches)
    patches = []
    for p in range(n_patches):
        shp = list(full_shape)
        shp[split_dim] = base + (1 if p < rem else 0)
        x = torch.randn(shp, generator=g, dtype=torch.float32) + float(patch_means[p])
        patches.append(x.to(TORCH_DTYPES[dtype]).contiguous())
    C = full_shape[1]
    gamma = (1.0 + 0.1 * torch.randn(C, generator=g, dtype=torch.float64)).to(TORCH_DTYPES[dtype])
    beta = (0.1 * torch.randn(C, generator=g, dtype=torch.float64)).to(TORCH_DTYPES[dtype])
    return patches, gamma, beta


def normal_tensor(seed: int, shape: Sequence[int], dtype: str) -> torch.Tensor:
    """i.i.d. N(0, 1) of ``shape``, drawn in float32 and cast."""
    g = _gen(seed)
    return torch.randn(list(shape), generator=g, dtype=torch.float32).to(TORCH_DTYPES[dtype]).contiguous()
