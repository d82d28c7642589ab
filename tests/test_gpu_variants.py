"""Two other builds of the same library, each run through the GPU parity tests
of the kernels it changes (in a child pytest whose binding loads that build
through TILEBLEND_LIB):

* the bounds-checked build (TB_DEBUG_BOUNDS=1): the stitch (both 2D/3D paths
  and the shard calls), the normalised-ramp stitch, the Patchify split and
  patch gather, and the halo pack check every computed tile index and every
  address before they read or write it; a check that fails records
  TB_DEV_OUT_OF_BOUNDS in the device status word (no trap) and skips the
  access.  Every full-size workload must stay bit-exact (or within its
  tolerance) and the word must read 0 at the end (the stitch file's last
  test);
* the TMA build (TB_STITCH_TMA=1): the stitch stages each piece's source
  rectangles with tensor copies instead of the per-thread cp.async rings; it
  must be bit-exact on every stitch and shard test as well;
* a GroupNorm build that cuts every statistics unit into 3 parts
  (TB_GN_FORCE_PARTS=3): records 3 to 7 of each unit are then empty and
  filled by the part CTAs in turn; the GroupNorm tests must still pass.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

VARIANTS = {
    "debug_bounds": (["TB_DEBUG_BOUNDS=1"], ["tests/test_gpu_patchify.py", "tests/test_gpu_ramp.py",
                                              "tests/test_gpu_shard.py", "tests/test_gpu_stitch.py"]),
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
