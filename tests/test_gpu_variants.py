"""Other builds of the same library, each run through the GPU parity tests
of the kernels it changes (in a child pytest whose binding loads that build
through TILEBLEND_LIB):

* the bounds-checked build (TB_DEBUG_BOUNDS=1): the stitch (both 2D/3D paths
  and the shard calls), the normalised-ramp stitch, the Patchify split and
  patch gather, the halo pack and the GroupNorm statistics and apply check
  every computed tile index, record index and address before they read or
  write it; a check that fails records
  TB_DEV_OUT_OF_BOUNDS in the device status word (no trap) and skips the
  access.  Every full-size workload must stay bit-exact (or within its
  tolerance) and the word must read 0 at the end (the stitch file's last
  test);
* the TMA build (TB_STITCH_TMA=1): the stitch stages each piece's source
  rectangles with tensor copies instead of the per-thread cp.async rings; it
  must be bit-exact on every stitch and shard test as well;
* a GroupNorm build that cuts every statistics unit into 3 parts
  (TB_GN_FORCE_PARTS=3): records 3 to 7 of each unit are then empty and
  filled by the part CTAs in turn; the GroupNorm tests must still pass;
* a GroupNorm build whose activation runs one element at a time
  (TB_GN_APPLY_PACKED=0): its outputs must equal the product build's bit for
  bit.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

VARIANTS = {
    "debug_bounds": (["TB_DEBUG_BOUNDS=1"], ["tests/test_gpu_patchify.py", "tests/test_gpu_ramp.py",
                                              "tests/test_gpu_shard.py", "tests/test_gpu_groupnorm.py",
                                              "tests/test_gpu_graph.py", "tests/test_gpu_stitch.py"]),
    "tma": (["TB_STITCH_TMA=1"], ["tests/test_gpu_shard.py", "tests/test_gpu_stitch.py"]),
    "gn_parts3": (["TB_GN_FORCE_PARTS=3"], ["tests/test_gpu_groupnorm.py", "tests/test_zz_no_alloc.py"]),
}


@pytest.mark.gpu
@pytest.mark.parametrize("variant", list(VARIANTS))
def test_variant_build_passes_the_parity_tests(variant):
    from patch_groupnorm_gb300 import build
    defines, files = VARIANTS[variant]
    path = build.build(variant=variant, defines=defines)
    env = dict(os.environ, TILEBLEND_LIB=path)
    r = subprocess.run([sys.executable, "-m", "pytest", *files, "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "failed" not in r.stdout


# The GroupNorm apply of the product build computes the activation's fp32
# steps on element pairs (fma/mul/add.rn.f32x2); TB_GN_APPLY_PACKED=0 computes
# them one element at a time.  Each lane of a packed instruction rounds as the
# scalar instruction does, so both builds must write the same bits.
_APPLY_CHILD = r"""
import sys, torch
from patch_groupnorm_gb300 import tileblend as tb
out = {}
for dt in (torch.float32, torch.float16, torch.bfloat16):
    g = torch.Generator().manual_seed(7)
    x = torch.randn(2, 64, 40, 96, generator=g, dtype=torch.float64) * 2.0 + 0.5
    parts = [p.contiguous().to(dt).cuda() for p in torch.split(x, [16, 24], dim=2)]
    gamma = (1 + 0.2 * torch.randn(64, generator=g, dtype=torch.float64)).to(dt).cuda()
    beta = (0.3 * torch.randn(64, generator=g, dtype=torch.float64)).to(dt).cuda()
    rec = tb.new_partials(len(parts), 2, 8, parts[0].device)
    tb.tb_patch_gn_stats(parts, 8, rec)
    for silu in (True, False):
        outs = [torch.empty_like(p) for p in parts]
        tb.tb_patch_gn_apply(parts, outs, 8, rec, gamma, beta, 1e-6, silu)
        out["%s_%d" % (dt, silu)] = [o.cpu() for o in outs]
torch.cuda.synchronize()
torch.save(out, sys.argv[1])
"""


@pytest.mark.gpu
def test_packed_and_scalar_activation_write_the_same_bits(tmp_path):
    from patch_groupnorm_gb300 import build
    import torch
    libs = {"packed": build.build(), "scalar": build.build(variant="gn_scalar_act",
                                                           defines=["TB_GN_APPLY_PACKED=0"])}
    got = {}
    for name, path in libs.items():
        dst = str(tmp_path / (name + ".pt"))
        env = dict(os.environ, TILEBLEND_LIB=path)
        r = subprocess.run([sys.executable, "-c", _APPLY_CHILD, dst], cwd=ROOT, env=env, capture_output=True,
                           text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        got[name] = torch.load(dst)
    assert got["packed"].keys() == got["scalar"].keys() and len(got["packed"]) == 6
    for key, outs in got["packed"].items():
        for a, b in zip(outs, got["scalar"][key]):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), key
