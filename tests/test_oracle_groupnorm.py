"""Pins for the PatchGroupNorm oracle (oracle/groupnorm.py): the library
GroupNorm on the unsharded tensor, invariants of the pooled statistics, the
variance the synthetic recipe implies, and the two broken variants the
DistVAE page describes, which must fail."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import groupnorm as GN
from oracle import rounding as R
from patch_groupnorm_gb300 import synth


def _split(x: np.ndarray, dim: int, sizes):
    return [np.ascontiguousarray(p) for p in np.split(x, np.cumsum(sizes)[:-1], axis=dim)]


@pytest.mark.parametrize("shape,dim,sizes", [
    ((2, 8, 12, 10), 2, [3, 3, 3, 3]),        # 4D split on height
    ((1, 12, 6, 11), 3, [4, 4, 3]),           # 4D split on width, ragged
    ((2, 6, 3, 5, 8), 4, [2, 2, 2, 2]),       # 5D split on width
    ((1, 6, 4, 7, 3), 3, [4, 3]),             # 5D split on height, ragged
    ((3, 4, 9), 2, [9]),                      # one patch: plain GroupNorm
])
@pytest.mark.parametrize("silu", [True, False])
def test_matches_torch_group_norm_float64(shape, dim, sizes, silu):
    rng = np.random.default_rng(20)
    x = rng.standard_normal(shape) * 1.7 + 0.4
    C = shape[1]
    G = 2 if C % 4 else 4
    gamma, beta = rng.standard_normal(C), rng.standard_normal(C)
    patches = _split(x, dim, sizes)
    ours = GN.patch_group_norm(patches, G, gamma, beta, 1e-6, silu=silu)
    ref = F.group_norm(torch.from_numpy(x), G, torch.from_numpy(gamma), torch.from_numpy(beta), 1e-6)
    if silu:
        ref = F.silu(ref)
    got = np.concatenate(ours, axis=dim)
    assert np.abs(got - ref.numpy()).max() < 1e-12


def test_variance_is_shift_invariant():
    rng = np.random.default_rng(21)
    x = rng.standard_normal((1, 8, 16, 16))
    patches = _split(x, 2, [4, 4, 4, 4])
    m0, v0 = GN.group_stats(patches, 4)
    m1, v1 = GN.group_stats([p + 3.0 for p in patches], 4)
    assert np.allclose(m1, m0 + 3.0, rtol=0, atol=1e-12)
    assert np.abs(v1 / v0 - 1).max() < 1e-12


def test_offsetting_one_patch_adds_the_between_patch_term():
    # law of total variance: var = mean of within-patch variances (weighted)
    # + weighted variance of the patch means about the pooled mean
    rng = np.random.default_rng(22)
    x = rng.standard_normal((1, 4, 10, 6))
    sizes = [4, 3, 3]
    patches = _split(x, 2, sizes)
    patches[1] = patches[1] + 2.5
    mean, var = GN.group_stats(patches, 2)
    cnt, pm, pm2 = GN.patch_partials(patches, 2)
    n = cnt.sum(axis=0)
    mu = (cnt * pm).sum(axis=0) / n
    expect = (pm2.sum(axis=0) + (cnt * (pm - mu) ** 2).sum(axis=0)) / n
    assert np.allclose(mean, mu, rtol=0, atol=1e-13)
    assert np.allclose(var, expect, rtol=1e-12, atol=0)


def test_patch_partials_match_numpy_mean_and_var():
    rng = np.random.default_rng(23)
    x = rng.standard_normal((2, 6, 5, 7)) + 1.0
    patches = _split(x, 3, [3, 4])
    cnt, pm, pm2 = GN.patch_partials(patches, 3)
    for p, patch in enumerate(patches):
        for n in range(2):
            for g in range(3):
                s = patch[n, 2 * g:2 * g + 2].ravel()
                assert cnt[p, n, g] == s.size
                assert abs(pm[p, n, g] - np.mean(s)) < 1e-14
                assert abs(pm2[p, n, g] - np.var(s) * s.size) < 1e-12


def test_synthetic_patch_means_give_pooled_variance_six():
    # patches ~ N(mu_p, 1), mu_p = -3, -1, 1, 3 in equal shares: the pooled
    # variance is 1 + mean(mu_p^2) = 1 + 5 = 6 and the pooled mean 0, up to
    # sampling error; the per-patch-mean variant only sees the within part.
    patches, _, _ = synth.groupnorm_patches(5, (1, 64, 64, 64), 2, 4, (-3, -1, 1, 3), "f32")
    pn = [p.numpy() for p in patches]
    mean, var = GN.group_stats(pn, 8)
    assert np.abs(mean).max() < 0.02
    assert np.abs(var - 6.0).max() < 0.05
    _, var_bad = GN.group_stats(pn, 8, variant="per_patch_mean")
    assert np.abs(var_bad - 1.0).max() < 0.05


def _bf16_ulp(v):
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    return 2.0 ** (e - 7)


@pytest.mark.parametrize("variant", ["per_patch_mean", "bessel"])
def test_broken_variants_fail_the_tolerance(variant):
    # a case built so that either mistake shows: patch means far apart, and
    # groups small enough that Bessel's n/(n-1) is visible in bf16.
    patches, gamma, beta = synth.groupnorm_patches(6, (1, 8, 8, 4), 2, 4, (-3, -1, 1, 3), "bf16")
    pn = [R.storage_to_f64(p.view(torch.int16).numpy().view(np.uint16), "bf16") for p in patches]
    g = R.storage_to_f64(gamma.view(torch.int16).numpy().view(np.uint16), "bf16")
    b = R.storage_to_f64(beta.view(torch.int16).numpy().view(np.uint16), "bf16")
    good = np.concatenate([R.storage_to_f64(R.round_f64(o, "bf16"), "bf16")
                           for o in GN.patch_group_norm(pn, 4, g, b, 1e-6)], axis=2)
    bad = np.concatenate([R.storage_to_f64(R.round_f64(o, "bf16"), "bf16")
                          for o in GN.patch_group_norm(pn, 4, g, b, 1e-6, variant=variant)], axis=2)
    assert (np.abs(bad - good) > _bf16_ulp(good)).any()


def test_broken_variants_agree_with_pooled_when_they_should():
    # one patch and a huge count: per-patch mean IS the pooled mean, and the
    # Bessel factor is within 1e-6 -- the variants differ only where the page
    # says they do.
    rng = np.random.default_rng(24)
    x = rng.standard_normal((1, 4, 300, 300))
    _, v = GN.group_stats([x], 2)
    _, v1 = GN.group_stats([x], 2, variant="per_patch_mean")
    _, v2 = GN.group_stats([x], 2, variant="bessel")
    assert np.allclose(v, v1, rtol=1e-12)
    n = 2 * 300 * 300
    assert np.allclose(v2, v * n / (n - 1), rtol=1e-12)
