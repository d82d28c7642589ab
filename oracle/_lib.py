"""ctypes handle on the oracle's C library.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).
"""
import ctypes

from . import build as _build

_LIB = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        L = ctypes.CDLL(_build.build())
        i64, i32p, vp = ctypes.c_int64, ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p
        L.orc_stitch.restype = ctypes.c_int
        L.orc_stitch.argtypes = [ctypes.c_int, i64, i32p, i32p, i32p, i32p, i32p, i32p,
                                 ctypes.POINTER(vp), vp]
        for name in ("orc_f32_to_f16", "orc_f32_to_bf16"):
            getattr(L, name).restype = ctypes.c_uint16
            getattr(L, name).argtypes = [ctypes.c_float]
        for name in ("orc_f64_to_f16", "orc_f64_to_bf16"):
            getattr(L, name).restype = ctypes.c_uint16
            getattr(L, name).argtypes = [ctypes.c_double]
        for name in ("orc_f16_value", "orc_bf16_value"):
            getattr(L, name).restype = ctypes.c_double
            getattr(L, name).argtypes = [ctypes.c_uint16]
        for name in ("orc_f32_to_f16_array", "orc_f32_to_bf16_array", "orc_f64_to_f16_array",
                     "orc_f64_to_bf16_array", "orc_f16_to_f64_array", "orc_bf16_to_f64_array"):
            getattr(L, name).restype = None
            getattr(L, name).argtypes = [vp, vp, i64]
        _LIB = L
    return _LIB
