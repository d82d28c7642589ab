"""The no-allocation PatchGroupNorm entry point (tb_patch_group_norm_noalloc).

It serves callers that cannot allocate device memory themselves (a host
framework that owns every allocation, a latency-critical path that must not
call cudaMalloc): the partial statistics live in a fixed scratch array inside
the library.  These tests call it through the C ABI.  It runs the same two
kernels as the two-call path with a caller-provided partials buffer, with the
same arguments, so its output must be identical bit for bit; they check that
on two calls in a row with different inputs (the scratch array keeps the
previous call's contents), compare one result with the float64 oracle, and
probe the size limit at and just past it.  This file is collected last and
also passes when run on its own.
"""
import pytest
import torch

from patch_groupnorm_gb300 import synth
from tests.tolerance import gn_violation

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tbl():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from patch_groupnorm_gb300 import build
    build.build()
    from patch_groupnorm_gb300 import tileblend
    return tileblend


def _inputs(seed, shape, split_dim, means):
    patches, gamma, beta = synth.groupnorm_patches(seed, shape, split_dim, len(means), means, "bf16")
    return patches, gamma, beta


def _two_call(tbl, patches, G, gamma, beta):
    ref = [torch.empty_like(p) for p in patches]
    partials = tbl.new_partials(len(patches), patches[0].shape[0], G)
    tbl.tb_patch_gn_stats(patches, G, partials)
    tbl.tb_patch_gn_apply(patches, ref, G, partials, gamma, beta, 1e-6, True)
    return ref


def test_noalloc_matches_the_two_call_path_on_consecutive_calls(tbl):
    cases = [
        (21, (1, 128, 64, 96), 2, (-3.0, -1.0, 1.0, 3.0), 32),   # first call on this device
        (22, (2, 64, 6, 20, 52), 4, (2.0, -2.0), 16),            # second call: other shape and patch count
    ]
    for k, (seed, shape, dim, means, G) in enumerate(cases):
        host, gamma, beta = _inputs(seed, shape, dim, means)
        patches = [p.cuda() for p in host]
        g, b = gamma.cuda(), beta.cuda()
        ref = _two_call(tbl, patches, G, g, b)
        got = [torch.full_like(p, float("nan")) for p in patches]
        tbl.tb_patch_group_norm_noalloc(patches, got, G, g, b, 1e-6, True)
        torch.cuda.synchronize()
        for o, r in zip(got, ref):
            assert torch.equal(o.view(torch.int16), r.view(torch.int16))
        if k == 0:
            assert gn_violation([o.cpu() for o in got], host, gamma, beta, G, 1e-6, True, "bf16") <= 1.0


def test_noalloc_at_its_limit_and_just_past_it(tbl):
    # room for P * N * G <= 65536 / TB_GN_PARTS = 8192 (patch, sample, group)
    # units: 2 patches x 64 samples x 64 groups fills it exactly
    limit = tbl.TB_NOALLOC_MAX_PARTIALS // tbl.TB_GN_PARTS
    assert 2 * 64 * 64 == limit
    x = synth.normal_tensor(23, (64, 64, 2, 8), "bf16").cuda()
    patches = [x[:, :, :1].contiguous(), x[:, :, 1:].contiguous() + 1.0]
    ref = _two_call(tbl, patches, 64, None, None)
    got = [torch.empty_like(p) for p in patches]
    tbl.tb_patch_group_norm_noalloc(patches, got, 64, None, None, 1e-6, True)
    torch.cuda.synchronize()
    for o, r in zip(got, ref):
        assert torch.equal(o.view(torch.int16), r.view(torch.int16))
    # one unit more (3 patches x 2731 samples x 1 group = 8193) is refused
    assert 3 * 2731 == limit + 1
    y = [torch.zeros((2731, 1, 4), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    outs = [torch.empty_like(p) for p in y]
    with pytest.raises(tbl.TileBlendError) as e:
        tbl.tb_patch_group_norm_noalloc(y, outs, 1, None, None, 1e-6, True)
    assert e.value.status == tbl.TB_ERR_UNSUPPORTED


def test_noalloc_rejects_sizes_beyond_its_scratch(tbl):
    # P * N * G = 2 * 1024 * 64 units, far past the 8192 the scratch holds
    patches = [torch.zeros((1024, 64, 1), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    outs = [torch.empty_like(p) for p in patches]
    with pytest.raises(tbl.TileBlendError) as e:
        tbl.tb_patch_group_norm_noalloc(patches, outs, 64, None, None, 1e-6, True)
    assert e.value.status == tbl.TB_ERR_UNSUPPORTED
