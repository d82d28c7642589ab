"""GPU parity of tb_patchify / tb_gather_patches against the numpy oracle
(oracle/patchify.py).  Both are copies, so the bar is bit-exact: tensors are
compared as their integer bit patterns.  Cases cover every chunk width the
kernel picks (16, 8, 4, 2 and 1 bytes), ragged and empty bands, padded
transfer slots, sizes the band rule would not produce, and the full-size
activations the benchmark times."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import patchify as PF
from patch_groupnorm_gb300 import synth
from patch_groupnorm_gb300 import workloads as W
from tests.tolerance import violation

pytestmark = pytest.mark.gpu

BITS = {torch.float32: torch.int32, torch.float16: torch.int16, torch.bfloat16: torch.int16}
NAMES = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


@pytest.fixture(scope="module")
def tbl():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from patch_groupnorm_gb300 import build
    build.build()
    from patch_groupnorm_gb300 import tileblend
    return tileblend


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(BITS[t.dtype]).cpu().numpy()


def _roundtrip(tbl, x, axis, factor, ranks, slot=0):
    xb = _bits(x)
    want = PF.patchify(xb, axis, factor, ranks)
    sizes = [p.shape[axis] for p in want]
    if slot:
        # pre-fill the slots so untouched padding is visible
        shapes = []
        for s in sizes:
            sh = list(x.shape)
            sh[axis] = slot
            shapes.append(sh)
        bufs = [torch.full(sh, -7.0, dtype=x.dtype, device="cuda") for sh in shapes]
        got = tbl.tb_patchify(x, axis, factor, ranks, patches=bufs, slot=slot)
    else:
        got = tbl.tb_patchify(x, axis, factor, ranks)
    torch.cuda.synchronize()
    for p, (g, w, s) in enumerate(zip(got, want, sizes)):
        gb = _bits(g)
        if slot:
            band = np.take(gb, np.arange(s), axis=axis)
            assert np.array_equal(band, w), "patch %d" % p
            pad = np.take(gb, np.arange(s, slot), axis=axis)
            sentinel = _bits(torch.tensor([-7.0], dtype=x.dtype))[0]
            assert (pad == sentinel).all(), "patch %d: padding written" % p
        else:
            assert gb.shape == w.shape and np.array_equal(gb, w), "patch %d" % p
    if slot:
        # garbage in the padding must not reach the result
        for g, s in zip(got, sizes):
            g.narrow(axis, s, slot - s).fill_(1e4)
    back = tbl.tb_gather_patches(got, sizes, axis, slot=slot)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(back), xb)
    if slot:
        assert np.array_equal(_bits(back), PF.gather_padded([_bits(g) for g in got], sizes, axis))
    else:
        assert np.array_equal(_bits(back), PF.gather_patches(want, axis))


CASES = [
    # shape, axis, factor, ranks, dtype          chunk width picked
    ((1, 5, 6, 40), 3, 8, 3, torch.bfloat16),    # 16 B: runs 32, 32, 16 B
    ((2, 3, 15, 7), 2, 1, 2, torch.float32),     # 4 B: 8 + 7 rows of 7 floats (the page's 15 over 2)
    ((1, 4, 16, 9), 2, 1, 3, torch.float16),     # 2 B: 6 + 5 + 5 rows (the page's 16 over 3)
    ((1, 2, 3, 10, 12), 4, 4, 3, torch.bfloat16),  # 8 B: 4-column runs
    ((1, 2, 3, 10, 13), 4, 1, 4, torch.float16),   # 2 B: 4, 3, 3, 3 columns
    ((64, 64, 3, 2), 2, 1, 3, torch.bfloat16),     # 4 B runs, one chunk each
    ((2, 24, 5), 1, 8, 5, torch.float32),          # more ranks than bands: two empty patches
    ((40, 7, 3), 0, 8, 3, torch.float16),          # split on the leading axis
    ((4096,), 0, 16, 7, torch.bfloat16),           # one axis
    ((3, 6, 256, 8), 2, 2, 64, torch.float32),     # the largest rank count
    ((3, 6, 16, 40), 2, 16, 1, torch.bfloat16),    # one rank: a plain copy
    ((2, 3, 37, 1000), 2, 1, 5, torch.bfloat16),   # many CTAs per patch, ragged tail
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_small_cases_roundtrip_bit_exact(tbl, case):
    shape, axis, factor, ranks, dt = case
    x = synth.normal_tensor(sum(shape) + ranks, shape, NAMES[dt]).cuda()
    _roundtrip(tbl, x, axis, factor, ranks)


@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[6]], ids=["16B", "2B", "empty"])
def test_padded_slots_leave_padding_untouched_and_are_sliced_on_gather(tbl, case):
    shape, axis, factor, ranks, dt = case
    x = synth.normal_tensor(sum(shape) + 2 * ranks, shape, NAMES[dt]).cuda()
    largest = max(PF.band_sizes(shape[axis], factor, ranks))
    _roundtrip(tbl, x, axis, factor, ranks, slot=largest + factor)


def test_gather_takes_any_sizes(tbl):
    sizes = [5, 0, 9, 1, 17]
    parts = [synth.normal_tensor(10 + i, (2, 3, s, 33), "bf16").cuda() for i, s in enumerate(sizes)]
    out = tbl.tb_gather_patches(parts, sizes, 2)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), PF.gather_patches([_bits(p) for p in parts], 2))


def test_byte_aligned_addresses_take_the_one_byte_path(tbl):
    # an f16 tensor at an odd byte address: only 1-byte chunks fit
    shape = (3, 20, 16)
    n = int(np.prod(shape))
    raw = torch.zeros(2 * n + 64, dtype=torch.uint8, device="cuda")
    src = synth.normal_tensor(5, shape, "f16")
    raw[1:1 + 2 * n] = src.view(torch.uint8).reshape(-1).cuda()
    outs = [torch.zeros(2 * n + 64, dtype=torch.uint8, device="cuda") for _ in range(3)]
    _, sizes = tbl.tb_patchify_layout(20, 4, 3)
    shp = (ctypes.c_int64 * 3)(*shape)
    ptrs = (ctypes.c_void_p * 3)(*[o.data_ptr() + 1 for o in outs])
    st = tbl._lib.tb_patchify(raw.data_ptr() + 1, tbl.TB_F16, 3, shp, 1, 4, 3, 0, ptrs, None)
    assert st == tbl.TB_OK
    torch.cuda.synchronize()
    want = PF.patchify(src.view(torch.int16).numpy(), 1, 4, 3)
    for o, w, s in zip(outs, want, sizes):
        got = o[1:1 + 2 * 3 * s * 16].cpu().numpy().view(np.int16).reshape(3, s, 16)
        assert np.array_equal(got, w)
        assert int(o[0]) == 0 and int(o[1 + 2 * 3 * s * 16:].sum()) == 0   # nothing outside the patch


@pytest.mark.parametrize("name", list(W.PATCHIFY))
def test_full_workloads(tbl, name):
    w = W.PATCHIFY[name]
    x = W.make_patchify_input(w).cuda()
    _roundtrip(tbl, x, w.axis, w.factor, w.ranks)


def test_split_feeds_patch_group_norm(tbl):
    # the split is the step in front of PatchGroupNorm: its ragged patches
    # normalise to the unsharded result (the page's 15 rows over 2 ranks)
    from oracle import groupnorm as GN
    from oracle import rounding as R
    x = synth.normal_tensor(21, (1, 64, 15, 24), "bf16")
    patches = tbl.tb_patchify(x.cuda(), 2, 1, 2)
    assert [p.shape[2] for p in patches] == [8, 7]
    outs = tbl.patch_group_norm(patches, 8, None, None, 1e-6, silu=True)
    whole = tbl.tb_gather_patches(outs, [8, 7], 2)
    torch.cuda.synchronize()
    exact = GN.patch_group_norm([x.double().numpy()], 8, None, None, 1e-6, silu=True)[0]
    assert violation(whole.double().cpu().numpy(), exact, "bf16") <= 1.0


def test_gather_writes_nothing_outside_its_output(tbl):
    shape = (2, 3, 37, 40)
    x = synth.normal_tensor(77, shape, "bf16").cuda()
    parts = tbl.tb_patchify(x, 2, 1, 5)
    guard = 4096
    buf = torch.full((x.numel() + 2 * guard,), 9.0, dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + x.numel()].view(shape)
    tbl.tb_gather_patches(parts, [p.shape[2] for p in parts], 2, out=out)
    torch.cuda.synchronize()
    assert (buf[:guard] == 9.0).all() and (buf[guard + x.numel():] == 9.0).all()
    assert np.array_equal(_bits(out), _bits(x))
