"""GPU parity of tb_patch_gn_stats / tb_patch_gn_apply against the float64
oracle.

Tolerances (tests/tolerance.py, derived from the arithmetic; the GroupNorm
is computed in fp32):
  * fp32 output: max-abs error 2e-5 against the exact (float64) value;
  * fp16 / bf16 output: at most 1 ulp of the storage type away from the
    oracle's once-rounded value, the ulp taken at max(|value|, floor) with
    floors 2^-12 (bf16) and 2^-9 (fp16): an absolute bound of 2^-19 near
    zero, where the output is a cancellation in x * a + b;
  * partial statistics: counts exact, means and M2 to 2e-5 relative.
"""
import numpy as np
import pytest
import torch

from oracle import groupnorm as GN
from oracle import rounding as R
from patch_groupnorm_gb300 import synth
from patch_groupnorm_gb300 import workloads as W
from tests.stitch_helpers import TORCH, to_storage
from tests.tolerance import gn_violation

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tbl():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from patch_groupnorm_gb300 import build
    build.build()
    from patch_groupnorm_gb300 import tileblend
    return tileblend


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def check_outputs(outs, patches, gamma, beta, G, eps, silu, dtype, variant="pooled"):
    """Max violation ratio (error / tolerance) of GPU outputs vs the oracle."""
    return gn_violation(outs, patches, gamma, beta, G, eps, silu, dtype, variant)


def run_gpu(tbl, patches, G, gamma, beta, eps, silu, inplace=False):
    dev = [p.cuda() for p in patches]
    part = tbl.new_partials(len(dev), dev[0].shape[0], G)
    g = None if gamma is None else gamma.cuda()
    b = None if beta is None else beta.cuda()
    outs = dev if inplace else [torch.empty_like(p) for p in dev]
    tbl.tb_patch_gn_stats(dev, G, part)
    tbl.tb_patch_gn_apply(dev, outs, G, part, g, b, eps, silu)
    torch.cuda.synchronize()
    return [o.cpu() for o in outs], part.cpu()


def _split(x: torch.Tensor, dim: int, sizes):
    return [p.contiguous() for p in torch.split(x, sizes, dim=dim)]


# --------------------------------------------------------------------------
# full workloads
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", list(W.GROUPNORM))
def test_full_workload_within_tolerance_and_not_the_broken_variants(tbl, name):
    w = W.GROUPNORM[name]
    patches, gamma, beta = W.make_groupnorm_inputs(w)
    outs, _ = run_gpu(tbl, patches, w.groups, gamma, beta, w.eps, True)
    with np.errstate(over="ignore"):
        assert check_outputs(outs, patches, gamma, beta, w.groups, w.eps, True, w.dtype) <= 1.0
        # the per-patch-mean mistake is far outside the bound
        assert check_outputs(outs, patches, gamma, beta, w.groups, w.eps, True, w.dtype,
                             variant="per_patch_mean") > 4.0


# --------------------------------------------------------------------------
# statistics
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_partials_match_oracle(tbl, dtype):
    patches, _, _ = synth.groupnorm_patches(3, (2, 24, 37, 16), 2, 3, (-3.0, 0.5, 2.0), dtype)
    _, part = run_gpu(tbl, patches, 6, None, None, 1e-6, True)
    part = part.view(-1, tbl.TB_GN_PARTS, 2).numpy()
    cnt = part[..., 0].astype(np.float64)
    packed = np.ascontiguousarray(part[..., 1]).view(np.float32).reshape(part.shape[0], tbl.TB_GN_PARTS, 2)
    mean, m2 = packed[..., 0].astype(np.float64), packed[..., 1].astype(np.float64)
    # merge each unit's parts: pooled count, mean, and M2 about the pooled mean
    n = cnt.sum(axis=1)
    mu = (cnt * mean).sum(axis=1) / n
    M2 = (m2 + cnt * (mean - mu[:, None]) ** 2).sum(axis=1)
    assert ((cnt > 0) | ((mean == 0) & (m2 == 0))).all()      # unused parts are empty records
    oc, om, om2 = GN.patch_partials([_f64(p) for p in patches], 6)
    assert np.array_equal(n, oc.reshape(-1))
    assert np.abs(mu - om.reshape(-1)).max() <= 2e-5 * np.maximum(1, np.abs(om)).max()
    assert np.abs(M2 / om2.reshape(-1) - 1).max() <= 2e-5


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_ragged_patches_with_an_empty_one_in_the_middle(tbl, dtype):
    # 768 units of 240-272 chunks (16 bytes) over ragged patches, one of them
    # empty and between the others: every record of the empty patch's units
    # is empty, the counts of each unit add up, and the pooled statistics and
    # outputs match the oracle.
    vec = 4 if dtype == "f32" else 8
    heights = [30, 0, 34, 32, 33, 31]
    g = torch.Generator().manual_seed(240)
    x = torch.randn(4, 64, sum(heights), 32 * 8 // vec, generator=g, dtype=torch.float64) * 1.3
    parts = _split(x, 2, heights)
    parts = [(p + m).to(TORCH[dtype]) for p, m in zip(parts, [-2.0, 0.0, 2.5, -1.0, 1.0, 3.0])]
    G = 32
    gamma = (1 + 0.1 * torch.randn(64, generator=g, dtype=torch.float64)).to(TORCH[dtype])
    beta = (0.1 * torch.randn(64, generator=g, dtype=torch.float64)).to(TORCH[dtype])
    outs, part = run_gpu(tbl, parts, G, gamma, beta, 1e-6, True)
    with np.errstate(over="ignore"):
        assert check_outputs(outs, parts, gamma, beta, G, 1e-6, True, dtype) <= 1.0
    part = part.view(-1, tbl.TB_GN_PARTS, 2).numpy()
    cnt = part[..., 0]
    packed = np.ascontiguousarray(part[..., 1]).view(np.float32).reshape(part.shape[0], tbl.TB_GN_PARTS, 2)
    assert ((cnt > 0) | ((packed[..., 0] == 0) & (packed[..., 1] == 0))).all()
    oc, om, om2 = GN.patch_partials([_f64(p) for p in parts], G)
    assert np.array_equal(cnt.sum(axis=1), oc.reshape(-1))
    assert (cnt.reshape(6, -1)[1] == 0).all()
    c64 = cnt.astype(np.float64)
    mean, m2 = packed[..., 0].astype(np.float64), packed[..., 1].astype(np.float64)
    n = c64.sum(axis=1)
    keep = n > 0
    mu = (c64 * mean).sum(axis=1)[keep] / n[keep]
    M2 = (m2[keep] + c64[keep] * (mean[keep] - mu[:, None]) ** 2).sum(axis=1)
    om, om2 = om.reshape(-1)[keep], om2.reshape(-1)[keep]
    assert np.abs(mu - om).max() <= 2e-5 * np.maximum(1, np.abs(om)).max()
    assert np.abs(M2 / om2 - 1).max() <= 2e-5


def test_stats_deterministic(tbl):
    patches, _, _ = synth.groupnorm_patches(4, (1, 64, 96, 96), 3, 4, (-3, -1, 1, 3), "bf16")
    _, a = run_gpu(tbl, patches, 32, None, None, 1e-6, False)
    _, b = run_gpu(tbl, patches, 32, None, None, 1e-6, False)
    assert torch.equal(a, b)


# --------------------------------------------------------------------------
# small cases: dtypes, ragged and unaligned patches, options
# --------------------------------------------------------------------------

CASES = [
    # full shape, split dim, patch sizes along it
    ((1, 32, 24, 40), 2, [6, 6, 6, 6]),          # 4D split on height
    ((2, 16, 10, 33), 3, [9, 8, 8, 8]),          # 4D split on width, ragged, odd rows (element path)
    ((1, 24, 5, 12, 16), 4, [4, 4, 4, 4]),       # 5D split on width
    ((1, 12, 3, 7, 9), 3, [4, 3]),               # 5D split on height, ragged, odd
    ((3, 8, 64), 2, [64]),                       # one patch: plain GroupNorm
]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[0])))
def test_small_cases(tbl, dtype, case):
    shape, dim, sizes = case
    g = torch.Generator().manual_seed(sum(shape))
    x = torch.randn(shape, generator=g, dtype=torch.float64) * 1.5
    # patch means far apart
    parts = _split(x, dim, sizes)
    parts = [(p + m).to(TORCH[dtype]) for p, m in zip(parts, [-3.0, 3.0, -1.0, 1.0])]
    C = shape[1]
    G = 4
    gamma = (1 + 0.1 * torch.randn(C, generator=g, dtype=torch.float64)).to(TORCH[dtype])
    beta = (0.1 * torch.randn(C, generator=g, dtype=torch.float64)).to(TORCH[dtype])
    for silu in (True, False):
        outs, _ = run_gpu(tbl, parts, G, gamma, beta, 1e-6, silu)
        with np.errstate(over="ignore"):
            assert check_outputs(outs, parts, gamma, beta, G, 1e-6, silu, dtype) <= 1.0


def test_no_affine_and_in_place(tbl):
    patches, _, _ = synth.groupnorm_patches(8, (1, 64, 32, 48), 2, 4, (-3, -1, 1, 3), "bf16")
    keep = [p.clone() for p in patches]
    outs, _ = run_gpu(tbl, patches, 8, None, None, 1e-5, True, inplace=True)
    with np.errstate(over="ignore"):
        assert check_outputs(outs, keep, None, None, 8, 1e-5, True, "bf16") <= 1.0


def test_empty_patch_and_empty_batch(tbl):
    a = torch.randn(1, 8, 0, 16, dtype=torch.float32)
    b = torch.randn(1, 8, 12, 16, dtype=torch.float32) + 2
    outs, part = run_gpu(tbl, [a, b], 2, None, None, 1e-6, True)
    assert check_outputs(outs[1:], [b], None, None, 2, 1e-6, True, "f32") <= 1.0
    assert (part.view(2, -1, 2)[0, :, 0] == 0).all()
    # N == 0: nothing launched
    e = torch.empty(0, 8, 4, 4, device="cuda")
    part = tbl.new_partials(1, 0, 2)
    tbl.tb_patch_gn_stats([e], 2, part)
    tbl.tb_patch_gn_apply([e], [e], 2, part, None, None, 1e-6, True)
    torch.cuda.synchronize()


def test_large_group_spans_several_ctas(tbl):
    # one big group per sample: every unit is split over several CTAs, each
    # writing its own part record
    patches, gamma, beta = synth.groupnorm_patches(9, (1, 8, 512, 512), 2, 2, (-3, 3), "bf16")
    outs, _ = run_gpu(tbl, patches, 1, gamma, beta, 1e-6, True)
    with np.errstate(over="ignore"):
        assert check_outputs(outs, patches, gamma, beta, 1, 1e-6, True, "bf16") <= 1.0


def test_largest_patch_count(tbl):
    # 64 patches (the most one call takes), one height row each, ragged widths of data per group
    x = torch.randn(2, 16, 64, 24, generator=torch.Generator().manual_seed(64), dtype=torch.float64)
    parts = [(x[:, :, r:r + 1] + (r % 7 - 3)).to(torch.bfloat16) for r in range(64)]
    outs, part = run_gpu(tbl, parts, 4, None, None, 1e-6, True)
    assert part.numel() * 8 == 64 * 2 * 4 * tbl.TB_GN_PARTS * 16
    with np.errstate(over="ignore"):
        assert check_outputs(outs, parts, None, None, 4, 1e-6, True, "bf16") <= 1.0


def test_guard_bands_and_inputs_untouched(tbl):
    # outputs and partials sit between canary bands; inputs are read only
    patches, gamma, beta = synth.groupnorm_patches(65, (2, 32, 20, 36), 3, 3, (-3.0, 0.0, 3.0), "bf16")
    dev = [p.cuda() for p in patches]
    keep = [p.clone() for p in dev]
    guard = 4096
    bufs, outs = [], []
    for p in dev:
        buf = torch.full((p.numel() + 2 * guard,), 77.0, dtype=torch.bfloat16, device="cuda")
        bufs.append(buf)
        outs.append(buf[guard:guard + p.numel()].view(p.shape))
    P, N, G = len(dev), dev[0].shape[0], 4
    n_rec = P * N * G * tbl.TB_GN_PARTS
    pbuf = torch.full((2 * n_rec + 2 * guard,), -5, dtype=torch.int64, device="cuda")
    part = pbuf[guard:guard + 2 * n_rec].view(P, N, G, tbl.TB_GN_PARTS, 2)
    tbl.tb_patch_gn_stats(dev, G, part)
    tbl.tb_patch_gn_apply(dev, outs, G, part, gamma.cuda(), beta.cuda(), 1e-6, True)
    torch.cuda.synchronize()
    for buf, p in zip(bufs, dev):
        assert (buf[:guard] == 77.0).all() and (buf[guard + p.numel():] == 77.0).all()
    assert (pbuf[:guard] == -5).all() and (pbuf[guard + 2 * n_rec:] == -5).all()
    for p, k in zip(dev, keep):
        assert torch.equal(p, k)
    with np.errstate(over="ignore"):
        assert check_outputs([o.cpu() for o in outs], patches, gamma, beta, G, 1e-6, True, "bf16") <= 1.0
