"""IEEE-754 round-to-nearest-even into fp16 and bf16, and exact widening.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Written from the definition of the binary16 and bfloat16 formats (the
rounding the stitch's contract names: each product and each sum rounded to
the storage type); the arithmetic lives in ``stitch.c``.  Narrow values are
carried as their raw ``uint16`` bit patterns.
"""
import numpy as np

from ._lib import lib


def f32_to_f16_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_f16_array(x.ctypes.data, y.ctypes.data, x.size)
    return y


def f32_to_bf16_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_array(x.ctypes.data, y.ctypes.data, x.size)
    return y


def f64_to_f16_bits(x) -> np.ndarray:
    """One rounding, straight from double."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f64_to_f16_array(x.ctypes.data, y.ctypes.data, x.size)
    return y


def f64_to_bf16_bits(x) -> np.ndarray:
    """One rounding, straight from double."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f64_to_bf16_array(x.ctypes.data, y.ctypes.data, x.size)
    return y


def f16_bits_to_f64(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    y = np.empty(b.shape, dtype=np.float64)
    lib().orc_f16_to_f64_array(b.ctypes.data, y.ctypes.data, b.size)
    return y


def bf16_bits_to_f64(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    y = np.empty(b.shape, dtype=np.float64)
    lib().orc_bf16_to_f64_array(b.ctypes.data, y.ctypes.data, b.size)
    return y


def round_f64(x, dtype: str) -> np.ndarray:
    """Round float64 values once into ``dtype`` ('f32', 'f16', 'bf16', 'f64');
    returns raw storage (float32 / uint16 bits / float64)."""
    if dtype == "f64":
        return np.ascontiguousarray(x, dtype=np.float64)
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)  # numpy: IEEE RNE
    if dtype == "f16":
        return f64_to_f16_bits(x)
    if dtype == "bf16":
        return f64_to_bf16_bits(x)
    raise ValueError(dtype)


def storage_to_f64(s, dtype: str) -> np.ndarray:
    """Exact values of raw storage as float64."""
    if dtype in ("f32", "f64"):
        return np.asarray(s, dtype=np.float64)
    if dtype == "f16":
        return f16_bits_to_f64(s)
    if dtype == "bf16":
        return bf16_bits_to_f64(s)
    raise ValueError(dtype)
