"""CPU oracle for the tile stitch and PatchGroupNorm.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, deliberately
unoptimised restatement of what the method computes, used to check the CUDA
library.  Only the test suite, the package smoke check and the benchmark's
CPU-baseline leg may import it; the product path (``patch_groupnorm_gb300``)
never does, and the two share no code.

Modules
-------
geometry   stock tiled-decode grid geometry (tile origins, extents, clamped
           blend extents, crops and output offsets), in plain Python.
stitch     the literal in-place blend_t / blend_v / blend_h recurrence with
           crop and concatenation, in plain C (``stitch.c``) behind ctypes.
rounding   IEEE round-to-nearest-even into fp16 / bf16, from the same C file.
groupnorm  the unsharded GroupNorm (+ SiLU) in float64 numpy, and the two
           broken PatchGroupNorm variants described on the DistVAE page, kept
           as negative controls.
ramp       the normalised-ramp stitch of equally sized tiles, in float64.
patchify   the ragged band split of one axis among ranks (whole bands of
           the VAE's scale factor, the first ranks one band more) and the
           gather that reassembles the patches, in plain numpy.
"""
