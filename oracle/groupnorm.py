"""PatchGroupNorm oracle: the unsharded GroupNorm (+ SiLU) in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: the page "Add tiled VAE parallelism & extended model support"
(xDiT DistVAE PR #14), in the commit that fixes PatchGroupNorm: a patch-
parallel GroupNorm must reproduce what ``nn.GroupNorm`` computes on the whole,
unsharded tensor -- the group mean pooled over every patch, and the biased
variance (divided by the element count, no Bessel correction) taken about
that pooled mean.  The decoder blocks follow the norm with SiLU.

So the oracle never looks at patches separately for the statistics: for each
(sample n, group g) it gathers the group's elements from every patch and
applies the plain two-pass definition

    mu     = sum(x) / count
    var    = sum((x - mu)^2) / count
    z      = (x - mu) / sqrt(var + eps) * gamma[c] + beta[c]
    y      = z / (1 + exp(-z))            (if silu)

in float64; the caller rounds the result once into the storage type.

The same page describes the two mistakes the fix removed.  They are kept
here, selected by ``variant``, only as negative controls that the tests
require to FAIL the tolerance:

  'per_patch_mean'  each patch's squared deviations are taken about that
                    patch's own mean (the pooled mean still centres x);
  'bessel'          the pooled variance divided by count - 1 (torch.var's
                    default).
"""
from typing import List, Sequence, Tuple

import numpy as np

VARIANTS = ("pooled", "per_patch_mean", "bessel")


def _group_slices(patch: np.ndarray, n: int, g: int, cg: int) -> np.ndarray:
    return patch[n, g * cg:(g + 1) * cg].reshape(-1)


def group_stats(patches: Sequence[np.ndarray], G: int, variant: str = "pooled") -> Tuple[np.ndarray, np.ndarray]:
    """Per (n, g) mean and variance over the union of all patches; float64
    arrays of shape [N, G]."""
    if variant not in VARIANTS:
        raise ValueError(variant)
    N, C = patches[0].shape[:2]
    if C % G:
        raise ValueError("channels must divide into groups")
    cg = C // G
    mean = np.zeros((N, G))
    var = np.zeros((N, G))
    for n in range(N):
        for g in range(G):
            parts = [np.asarray(_group_slices(p, n, g, cg), dtype=np.float64) for p in patches]
            x = np.concatenate(parts)
            count = x.size
            mu = x.sum() / count
            if variant == "per_patch_mean":
                m2 = sum(((q - q.mean()) ** 2).sum() for q in parts if q.size)
                v = m2 / count
            elif variant == "bessel":
                v = ((x - mu) ** 2).sum() / (count - 1)
            else:
                v = ((x - mu) ** 2).sum() / count
            mean[n, g] = mu
            var[n, g] = v
    return mean, var


def patch_partials(patches: Sequence[np.ndarray], G: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Per patch p, sample n, group g: element count, the patch's own group
    mean and the sum of squared deviations about it.  Arrays [P, N, G]
    (counts int64, the rest float64)."""
    P = len(patches)
    N, C = patches[0].shape[:2]
    cg = C // G
    cnt = np.zeros((P, N, G), dtype=np.int64)
    mean = np.zeros((P, N, G))
    m2 = np.zeros((P, N, G))
    for p, patch in enumerate(patches):
        for n in range(N):
            for g in range(G):
                x = np.asarray(_group_slices(patch, n, g, cg), dtype=np.float64)
                cnt[p, n, g] = x.size
                if x.size:
                    mu = x.sum() / x.size
                    mean[p, n, g] = mu
                    m2[p, n, g] = ((x - mu) ** 2).sum()
    return cnt, mean, m2


def patch_group_norm(patches: Sequence[np.ndarray], G: int, gamma, beta, eps: float,
                     silu: bool = True, variant: str = "pooled") -> List[np.ndarray]:
    """GroupNorm of the unsharded tensor, returned patch by patch (float64).

    ``patches[p]`` is [N, C, *spatial_p]; ``gamma`` / ``beta`` are [C] or None
    (None means 1 / 0)."""
    N, C = patches[0].shape[:2]
    cg = C // G
    mean, var = group_stats(patches, G, variant)
    gam = np.ones(C) if gamma is None else np.asarray(gamma, dtype=np.float64)
    bet = np.zeros(C) if beta is None else np.asarray(beta, dtype=np.float64)
    outs = []
    for patch in patches:
        x = np.asarray(patch, dtype=np.float64)
        y = np.empty_like(x)
        for n in range(N):
            for c in range(C):
                g = c // cg
                z = (x[n, c] - mean[n, g]) / np.sqrt(var[n, g] + eps) * gam[c] + bet[c]
                if silu:
                    z = z / (1.0 + np.exp(-z))
                y[n, c] = z
        outs.append(y)
    return outs
