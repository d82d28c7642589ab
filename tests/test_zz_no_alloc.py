"""The no-allocation PatchGroupNorm entry point (tb_patch_group_norm_noalloc).

It serves callers that cannot allocate device memory themselves (a host
framework that owns every allocation, a latency-critical path that must not
call cudaMalloc): the partial statistics live in a fixed scratch array inside
the library.  These tests call it through the C ABI and compare its output
with the two-call path that uses a caller-provided partials buffer, within
the tolerance of the GroupNorm tests, on two calls in a row with different
inputs (the scratch array keeps the previous call's contents).  This file is
collected last and also passes when run on its own.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tbl():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from patch_groupnorm_gb300 import build
    build.build()
    from patch_groupnorm_gb300 import tileblend
    return tileblend


def _within_one_ulp(got: torch.Tensor, ref: torch.Tensor) -> bool:
    # same bound as the GroupNorm parity tests: 1 bf16 ulp taken at max(|v|, 2^-8)
    g = got.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -8))) - 7)
    return bool((np.abs(g - r) <= ulp).all())


def _inputs(seed, shape, split_dim, means):
    from patch_groupnorm_gb300 import synth
    patches, gamma, beta = synth.groupnorm_patches(seed, shape, split_dim, len(means), means, "bf16")
    return [p.cuda() for p in patches], gamma.cuda(), beta.cuda()


def test_noalloc_matches_the_two_call_path_on_consecutive_calls(tbl):
    cases = [
        (21, (1, 128, 64, 96), 2, (-3.0, -1.0, 1.0, 3.0), 32),   # first call on this device
        (22, (2, 64, 6, 20, 52), 4, (2.0, -2.0), 16),            # second call: other shape and patch count
    ]
    for seed, shape, dim, means, G in cases:
        patches, gamma, beta = _inputs(seed, shape, dim, means)
        ref = [torch.empty_like(p) for p in patches]
        partials = tbl.new_partials(len(patches), shape[0], G)
        tbl.tb_patch_gn_stats(patches, G, partials)
        tbl.tb_patch_gn_apply(patches, ref, G, partials, gamma, beta, 1e-6, True)
        got = [torch.full_like(p, float("nan")) for p in patches]
        tbl.tb_patch_group_norm_noalloc(patches, got, G, gamma, beta, 1e-6, True)
        torch.cuda.synchronize()
        for o, r in zip(got, ref):
            assert _within_one_ulp(o, r)


def test_noalloc_rejects_sizes_beyond_its_scratch(tbl):
    # P * N * G = 2 * 1024 * 64 > 65536 records
    patches = [torch.zeros((1024, 64, 1), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    outs = [torch.empty_like(p) for p in patches]
    with pytest.raises(tbl.TileBlendError) as e:
        tbl.tb_patch_group_norm_noalloc(patches, outs, 64, None, None, 1e-6, True)
    assert e.value.status == tbl.TB_ERR_UNSUPPORTED
