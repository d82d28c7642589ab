"""Build libtileblend.so for GB300 (sm_103a) with nvcc, in-tree.

The translation units are compiled in parallel and linked into
``patch_groupnorm_gb300/_build/libtileblend.so`` (static CUDA runtime, only
the C ABI of ``include/tileblend.h`` exported).  The stitch unit is built
with ``-fmad=false`` so that no multiply and add fuse: the stitch's rounding
contract rounds every product and sum separately.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libtileblend.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-I", INCLUDE, "-I", CSRC,
          "-Xcompiler", "-fPIC,-fvisibility=hidden,-ffp-contract=off"]
UNITS = {
    "tb_host.cpp": [],
    "tb_stitch.cu": ["-fmad=false"],
    "tb_groupnorm.cu": [],
    "tb_noalloc.cu": [],
    "tb_ramp.cu": [],
    "tb_patchify.cu": [],
    "tb_shard.cu": [],
    "tb_status.cu": [],
}
HEADERS = ["tb_internal.h"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def lib_path(variant: str = "") -> str:
    """Path of the library build `variant` ('' is the product build)."""
    return LIB if not variant else os.path.join(OUT_DIR, "libtileblend-%s.so" % variant)


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = [os.path.join(CSRC, u) for u in UNITS] + [os.path.join(CSRC, h) for h in HEADERS]
    deps.append(os.path.join(INCLUDE, "tileblend.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, variant: str = "", defines=()) -> str:
    """Compile and link the library if it is missing or out of date.

    `variant` with `defines` (preprocessor definitions such as
    "TB_DEBUG_BOUNDS=1") builds a separate library, libtileblend-<variant>.so,
    next to the product build; the binding loads it when the environment
    variable TILEBLEND_LIB names it."""
    path = lib_path(variant)
    if not force and not _stale(path):
        return path
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    tag = "%s%d" % (variant + "." if variant else "", os.getpid())
    dflags = ["-D" + d for d in defines]

    def compile_unit(unit):
        obj = os.path.join(OUT_DIR, unit.rsplit(".", 1)[0] + "." + tag + ".o")
        cmd = [nvcc, *ARCH, *COMMON, *dflags, *UNITS[unit], "-c", os.path.join(CSRC, unit), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (unit, r.stdout, r.stderr))
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(UNITS)) as pool:
        objs = list(pool.map(compile_unit, UNITS))
    tmp = path + "." + tag + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, path)
    for o in objs:
        os.remove(o)
    return path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
