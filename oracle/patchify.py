"""Ragged Patchify split and the patch gather, in plain numpy.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: the page "Add tiled VAE parallelism & extended model support"
(xDiT DistVAE PR #14), the commit that stops Patchify from padding the split
axis, and the commit that removes ``use_uniform_patch``:

  * the split axis is cut into bands whose extents are whole multiples of the
    factor by which the VAE narrows or widens that axis, so every band stays
    on the grid the strided convolutions step along;
  * when the band count does not divide evenly among the ranks, the ranks
    that come first get one band more; no rows are invented (no padding);
  * ``gather_patches`` first exchanges the patch sizes, then the payload;
    because a collective all-gather wants equal shapes, each patch is padded
    to the longest for the transfer and the padding is sliced off on the
    receiving side before the patches are concatenated in rank order.

Readings taken where the page is silent:
  * an axis extent that is not a whole number of bands is refused (the page
    only speaks of axes cut in whole bands);
  * with more ranks than bands, the trailing ranks get empty patches;
  * the padding's values are never read, so the oracle fills it with zeros
    and the tests fill it with garbage.
"""
from typing import List, Sequence, Tuple

import numpy as np


def band_sizes(extent: int, factor: int, ranks: int) -> List[int]:
    """Extent of each rank's patch along the split axis, in rank order."""
    if factor < 1 or ranks < 1 or extent < 0:
        raise ValueError("factor and ranks must be >= 1, extent >= 0")
    if extent % factor:
        raise ValueError("the axis is not a whole number of bands")
    bands = extent // factor
    each, extra = divmod(bands, ranks)
    return [(each + (1 if r < extra else 0)) * factor for r in range(ranks)]


def band_starts(sizes: Sequence[int]) -> List[int]:
    """Offset of each patch along the split axis (running sum of sizes)."""
    starts, at = [], 0
    for s in sizes:
        starts.append(at)
        at += s
    return starts


def patchify(x: np.ndarray, axis: int, factor: int, ranks: int) -> List[np.ndarray]:
    """The ranks' patches of ``x`` cut along ``axis`` (copies)."""
    sizes = band_sizes(x.shape[axis], factor, ranks)
    out = []
    for start, size in zip(band_starts(sizes), sizes):
        idx = [slice(None)] * x.ndim
        idx[axis] = slice(start, start + size)
        out.append(np.array(x[tuple(idx)], copy=True))
    return out


def pad_for_transfer(patch: np.ndarray, axis: int, slot: int) -> np.ndarray:
    """The sending side: ``patch`` zero-padded at the end of ``axis`` to
    ``slot`` (the longest patch), so every rank sends the same shape."""
    if patch.shape[axis] > slot:
        raise ValueError("slot shorter than the patch")
    shape = list(patch.shape)
    shape[axis] = slot
    out = np.zeros(shape, dtype=patch.dtype)
    idx = [slice(None)] * patch.ndim
    idx[axis] = slice(0, patch.shape[axis])
    out[tuple(idx)] = patch
    return out


def gather_patches(patches: Sequence[np.ndarray], axis: int) -> np.ndarray:
    """Concatenation of the patches in rank order along ``axis``."""
    return np.concatenate(list(patches), axis=axis)


def gather_padded(slots: Sequence[np.ndarray], sizes: Sequence[int], axis: int) -> np.ndarray:
    """The receiving side: every slot sliced to its patch's size along
    ``axis`` (the sizes exchanged first), then concatenated in rank order."""
    kept = []
    for slot, size in zip(slots, sizes):
        idx = [slice(None)] * slot.ndim
        idx[axis] = slice(0, size)
        kept.append(slot[tuple(idx)])
    return gather_patches(kept, axis)


def layout(extent: int, factor: int, ranks: int) -> Tuple[List[int], List[int]]:
    """(starts, sizes) of the ranks' bands."""
    sizes = band_sizes(extent, factor, ranks)
    return band_starts(sizes), sizes
