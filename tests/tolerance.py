"""Tolerances of the floating-point parity tests (GroupNorm, the ramp
stitch), derived from the arithmetic of an fp32 pipeline and from measured
worst errors on the full workloads.

* fp32 output: max-abs error 2e-5 against the exact (float64) value.
* fp16 / bf16 output: at most 1 ulp of the storage type away from the
  oracle's once-rounded value.  The ulp is taken at max(|value|, floor):
  near zero an output is the cancellation of x * a against b in fp32, whose
  absolute error (a few fp32 ulps of |b| plus the statistics' error times
  |x * a|) no longer shrinks with the value.  The floors, 2^-12 for bf16 and
  2^-9 for fp16, both give an absolute bound of 2^-19 (1.9e-6) there, ten
  times below the fp32 tolerance.
"""
import numpy as np
import torch

from oracle import groupnorm as GN
from oracle import rounding as R

F32_ABS = 2e-5
FLOOR = {"bf16": 2.0 ** -12, "f16": 2.0 ** -9}
MANT = {"bf16": 7, "f16": 10}


def ulp_bound(ref: np.ndarray, dtype: str) -> np.ndarray:
    """1 ulp of `dtype` at max(|ref|, floor)."""
    m = np.maximum(np.abs(ref), FLOOR[dtype])
    return 2.0 ** (np.floor(np.log2(m)) - MANT[dtype])


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def violation(got: np.ndarray, exact: np.ndarray, dtype: str) -> float:
    """Largest error / tolerance over the elements (<= 1 passes); `exact` is
    the float64 result, rounded here once into `dtype` for 16-bit types."""
    if got.size == 0:
        return 0.0
    if dtype == "f32":
        return float(np.abs(got - exact).max()) / F32_ABS
    ref = R.storage_to_f64(R.round_f64(exact, dtype), dtype)
    return float((np.abs(got - ref) / ulp_bound(ref, dtype)).max())


def gn_violation(outs, patches, gamma, beta, G, eps, silu, dtype, variant="pooled") -> float:
    """Worst violation of GPU GroupNorm outputs against the float64 oracle."""
    exact = GN.patch_group_norm([f64(p) for p in patches], G, None if gamma is None else f64(gamma),
                                None if beta is None else f64(beta), eps, silu=silu, variant=variant)
    return max(violation(f64(o), e, dtype) for o, e in zip(outs, exact))
