"""Shared helpers for the stitch tests: storage conversion between torch
tensors and the oracle's raw numpy form, and a brute-force replay of the
tiled-decode blend loops written with torch CPU tensor ops.

The replay restates the loops the page "[Proposal] Vectorize tiled VAE
blending while preserving rounding and CUDA graph replay" describes (blend_v,
blend_h, blend_t with clamped extents, in place, then crop and concatenate),
one row / column / frame at a time, with Python-double coefficients.  Its
rounding is torch's own arithmetic, which is the authority the page's parity
tests compare against; it shares nothing with the C oracle.
"""
import numpy as np
import torch

TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "f64": torch.float64}


def to_storage(t: torch.Tensor, dtype: str) -> np.ndarray:
    t = t.contiguous()
    if dtype in ("f16", "bf16"):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def from_storage(a: np.ndarray, dtype: str) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if dtype in ("f16", "bf16"):
        return torch.from_numpy(a.view(np.int16)).view(TORCH[dtype])
    return torch.from_numpy(a)


def _blend_v(a, b, blend_extent):
    e = min(a.shape[-2], b.shape[-2], blend_extent)
    for y in range(e):
        b[..., y, :] = a[..., -e + y, :] * (1 - y / e) + b[..., y, :] * (y / e)
    return b


def _blend_h(a, b, blend_extent):
    e = min(a.shape[-1], b.shape[-1], blend_extent)
    for x in range(e):
        b[..., :, x] = a[..., :, -e + x] * (1 - x / e) + b[..., :, x] * (x / e)
    return b


def _blend_t(a, b, blend_extent):
    e = min(a.shape[-3], b.shape[-3], blend_extent)
    for t in range(e):
        b[..., t, :, :] = a[..., -e + t, :, :] * (1 - t / e) + b[..., t, :, :] * (t / e)
    return b


def torch_replay_2d(tiles, blend_y, limit_y, blend_x, limit_x):
    rows = [[t.clone() for t in row] for row in tiles]
    out_rows = []
    for i, row in enumerate(rows):
        out_row = []
        for j, tile in enumerate(row):
            if i > 0:
                tile = _blend_v(rows[i - 1][j], tile, blend_y)
            if j > 0:
                tile = _blend_h(row[j - 1], tile, blend_x)
            out_row.append(tile[..., :limit_y, :limit_x])
        out_rows.append(torch.cat(out_row, dim=-1))
    return torch.cat(out_rows, dim=-2)


def torch_replay_3d(tiles, blend_t, limit_t, blend_y, limit_y, blend_x, limit_x):
    grid = [[[t.clone() for t in row] for row in plane] for plane in tiles]
    out_planes = []
    for k, plane in enumerate(grid):
        out_rows = []
        for i, row in enumerate(plane):
            out_row = []
            for j, tile in enumerate(row):
                if k > 0:
                    tile = _blend_t(grid[k - 1][i][j], tile, blend_t)
                if i > 0:
                    tile = _blend_v(plane[i - 1][j], tile, blend_y)
                if j > 0:
                    tile = _blend_h(row[j - 1], tile, blend_x)
                out_row.append(tile[..., :limit_t, :limit_y, :limit_x])
            out_rows.append(torch.cat(out_row, dim=-1))
        out_planes.append(torch.cat(out_rows, dim=-2))
    return torch.cat(out_planes, dim=-3)


def boxes(layout, scale):
    """(origin in output space, extent) of each tile along an axis, for the
    input generator; ``scale`` converts the latent origins."""
    return [(o * scale, L) for o, L in zip(layout.origins, layout.extents)]
