"""The tiled-decode stitch: blend recurrence, crop and concatenation.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Thin ctypes marshalling around ``orc_stitch`` in ``stitch.c``, which holds the
arithmetic (the page "[Proposal] Vectorize tiled VAE blending while
preserving rounding and CUDA graph replay", "Proposed scope": the blend
loops, their extent clamp, their in-place updates and their rounding of
each product separately).

Tiles are numpy arrays in raw storage form: float32 for 'f32', float64 for
'f64', and uint16 bit patterns for 'f16' / 'bf16'.
"""
import ctypes
from typing import List, Sequence

import numpy as np

from ._lib import lib
from .geometry import AxisLayout, single_axis

DTYPES = {"f32": (0, np.float32), "f16": (1, np.uint16), "bf16": (2, np.uint16), "f64": (3, np.float64)}


def _i32(values) -> ctypes.Array:
    return (ctypes.c_int32 * max(1, len(values)))(*values)


def stitch(tiles: Sequence, axes: Sequence[AxisLayout], dtype: str) -> np.ndarray:
    """Stitch a 2D grid (``axes = (ay, ax)``, ``tiles[i][j]`` of shape
    [B, C, Ly(i), Lx(j)]) or a 3D grid (``axes = (at, ay, ax)``,
    ``tiles[k][i][j]`` of shape [B, C, Lt(k), Ly(i), Lx(j)]).

    Returns the output [B, C, H, W] or [B, C, T, H, W] in raw storage form.
    """
    code, npdt = DTYPES[dtype]
    if len(axes) == 2:
        ay, ax = axes
        grid = [[list(row) for row in tiles]]
        at = None
    elif len(axes) == 3:
        at, ay, ax = axes
        grid = [[list(row) for row in plane] for plane in tiles]
    else:
        raise ValueError("2 or 3 axes")
    nt = len(grid)
    ny, nx = ay.n, ax.n
    flat: List[np.ndarray] = []
    B = C = None
    for k in range(nt):
        assert len(grid[k]) == ny
        for i in range(ny):
            assert len(grid[k][i]) == nx
            for j in range(nx):
                t = np.ascontiguousarray(grid[k][i][j], dtype=npdt)
                if at is None:
                    t = t[:, :, None]
                if B is None:
                    B, C = t.shape[0], t.shape[1]
                exp = (B, C, at.extents[k] if at else 1, ay.extents[i], ax.extents[j])
                if t.shape != exp:
                    raise ValueError(f"tile ({k},{i},{j}) has shape {t.shape}, expected {exp}")
                flat.append(t)
    if at is None:
        at_eff = single_axis(1)
    else:
        at_eff = at
    out = np.zeros((B, C, at_eff.out_extent, ay.out_extent, ax.out_extent), dtype=npdt)
    ptrs = (ctypes.c_void_p * len(flat))(*[t.ctypes.data for t in flat])
    rc = lib().orc_stitch(
        code, B * C, _i32([nt, ny, nx]), _i32(at_eff.extents), _i32(ay.extents), _i32(ax.extents),
        _i32([at_eff.blend_extent, ay.blend_extent, ax.blend_extent]),
        _i32([at_eff.row_limit, ay.row_limit, ax.row_limit]), ptrs, out.ctypes.data)
    if rc != 0:
        raise MemoryError("oracle stitch ran out of memory")
    if at is None:
        out = out[:, :, 0]
    return out
