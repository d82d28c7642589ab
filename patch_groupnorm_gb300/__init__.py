"""libtileblend: GB300-native tile stitching and PatchGroupNorm.

The compute lives in the C-ABI shared library ``libtileblend.so`` (CUDA
kernels for sm_103a, declared in ``include/tileblend.h``); ``tileblend``
is its thin Python binding.  ``synth`` draws seeded synthetic inputs.
"""
__all__ = ["tileblend", "synth"]
