"""CPU-only checks of libtileblend: it builds, loads, exports every call the
header declares, derives the same geometry as the oracle, and rejects bad
arguments on the host before touching a GPU."""
import ctypes
import json
import os
import random
import re

import pytest

from oracle.geometry import axis_layout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tileblend.h")


@pytest.fixture(scope="module")
def tbl():
    from patch_groupnorm_gb300 import build
    build.build()
    from patch_groupnorm_gb300 import tileblend
    return tileblend


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tb_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    assert set(_declared_functions()) >= {"tb_stitch2d", "tb_stitch3d", "tb_patch_gn_stats", "tb_patch_gn_apply"}


def test_library_exports_every_declared_symbol(tbl):
    lib = ctypes.CDLL(tbl.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) == set(tbl.EXPORTED)


def test_library_exports_nothing_else(tbl):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", tbl.LIB_PATH], capture_output=True, text=True).stdout
    ours = sorted(l.split()[-1] for l in out.splitlines() if l.split()[-1].startswith("tb_"))
    assert ours == _declared_functions()


def test_version(tbl):
    assert tbl.tb_version() >= 100


GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "geometry.json")))["cases"]


@pytest.mark.parametrize("case", GOLDEN, ids=[c["name"] for c in GOLDEN])
def test_layout_matches_golden(tbl, case):
    lay = tbl.tb_axis_layout(tbl.Axis(case["latent_extent"], case["latent_tile"], case["overlap"], case["scale"]))
    assert lay.extents == case["extents"]
    assert lay.blends == case["blends"]
    assert lay.kept == case["kept"]
    assert lay.out_extent == case["out_extent"]


def test_layout_matches_oracle_on_random_axes(tbl):
    rnd = random.Random(7)
    for _ in range(3000):
        tile = rnd.randint(1, 160)
        ov = rnd.choice([0.0, 0.125, 0.2, 0.25, 0.3, 1 / 3, 0.5, 0.6, 0.75, rnd.random() * 0.95])
        if int(tile * (1 - ov)) < 1:
            continue
        ext = rnd.randint(0, 40 * max(1, int(tile * (1 - ov))))
        scale = rnd.choice([1, 2, 4, 8, 16])
        be = rnd.choice([None, None, rnd.randint(0, 300)])
        rl = rnd.choice([None, None, rnd.randint(1, 900)])
        o = axis_layout(ext, tile, ov, scale, be, rl)
        if o.n > tbl.TB_MAX_TILES_PER_AXIS:
            continue
        if o.row_limit < 1:
            continue
        lay = tbl.tb_axis_layout(tbl.Axis(ext, tile, ov, scale, -1 if be is None else be, 0 if rl is None else rl))
        assert (lay.n, lay.extents, lay.blends, lay.kept, lay.out_extent) == \
               (o.n, o.extents, o.blends, o.kept, o.out_extent), (ext, tile, ov, scale, be, rl)
        assert lay.origins == [v * scale for v in o.origins]


@pytest.mark.parametrize("bad", [
    dict(latent_extent=-1), dict(latent_tile=0), dict(scale=0), dict(overlap=1.0), dict(overlap=-0.1),
    dict(overlap=float("nan")), dict(latent_tile=1, overlap=0.5),  # zero stride
    dict(blend_extent=600, row_limit=0),                           # derived row_limit < 1
])
def test_layout_rejects_bad_geometry(tbl, bad):
    kw = dict(latent_extent=128, latent_tile=64, overlap=0.25, scale=8, blend_extent=-1, row_limit=0)
    kw.update(bad)
    with pytest.raises(tbl.TileBlendError) as e:
        tbl.tb_axis_layout(tbl.Axis(**kw))
    assert e.value.status == tbl.TB_ERR_GEOMETRY


def test_layout_too_many_tiles_is_unsupported_and_reports_count(tbl):
    a = tbl.Axis(1000, 8, 0.5, 8).c()
    n = ctypes.c_int32(0)
    st = tbl._lib.tb_axis_layout(ctypes.byref(a), 0, ctypes.byref(n), None, None, None, None, None)
    assert st == tbl.TB_ERR_UNSUPPORTED and n.value == 250


# --- host-side validation of the compute calls: no GPU is touched -----------

def _stitch2d(tbl, dtype=0, B=1, C=3, ay=None, ax=None, H=1024, W=1024, tiles="ok", out=16):
    ay = ay or tbl.Axis(128, 64, 0.25, 8)
    ax = ax or tbl.Axis(128, 64, 0.25, 8)
    arr = (ctypes.c_void_p * 256)(*([16 * (k + 1) for k in range(256)])) if tiles == "ok" else tiles
    a_y, a_x = ay.c(), ax.c()
    return tbl._lib.tb_stitch2d(arr, dtype, B, C, ctypes.byref(a_y), ctypes.byref(a_x), out, H, W, None)


def test_stitch_rejects_before_launch(tbl):
    assert _stitch2d(tbl, dtype=7) == tbl.TB_ERR_DTYPE
    assert _stitch2d(tbl, H=1000) == tbl.TB_ERR_SHAPE
    assert _stitch2d(tbl, W=-1) == tbl.TB_ERR_SHAPE
    assert _stitch2d(tbl, B=-2) == tbl.TB_ERR_SHAPE
    assert _stitch2d(tbl, out=None) == tbl.TB_ERR_NULL
    assert _stitch2d(tbl, tiles=None) == tbl.TB_ERR_NULL
    nulls = (ctypes.c_void_p * 9)(*([16] * 8 + [None]))
    assert _stitch2d(tbl, tiles=nulls) == tbl.TB_ERR_NULL
    assert _stitch2d(tbl, ay=tbl.Axis(128, 64, 1.5, 8)) == tbl.TB_ERR_GEOMETRY
    # bands that reach each other (overlap 3/4): outside the closed form
    chain = tbl.Axis(128, 64, 0.75, 8)
    lay = axis_layout(128, 64, 0.75, 8)
    assert _stitch2d(tbl, ay=chain, H=lay.out_extent) == tbl.TB_ERR_UNSUPPORTED
    # nothing to do: no launch, success, even with null pointers
    assert _stitch2d(tbl, B=0, tiles=None, out=None) == tbl.TB_OK
    assert _stitch2d(tbl, ay=tbl.Axis(0, 64, 0.25, 8), H=0, tiles=None, out=None) == tbl.TB_OK


def test_stitch3d_rejects_before_launch(tbl):
    at, ay, ax = tbl.Axis(49, 16, 0.25, 1).c(), tbl.Axis(60, 32, 0.25, 8).c(), tbl.Axis(104, 32, 0.25, 8).c()
    arr = (ctypes.c_void_p * 75)(*([16] * 75))
    f = tbl._lib.tb_stitch3d
    assert f(arr, 2, 1, 3, None, ctypes.byref(ay), ctypes.byref(ax), 16, 49, 480, 832, None) == tbl.TB_ERR_NULL
    assert f(arr, 2, 1, 3, ctypes.byref(at), ctypes.byref(ay), ctypes.byref(ax), 16, 48, 480, 832, None) \
        == tbl.TB_ERR_SHAPE


def test_groupnorm_rejects_before_launch(tbl):
    ptrs = (ctypes.c_void_p * 4)(16, 32, 48, 64)
    sp = (ctypes.c_int64 * 4)(100, 100, 100, 100)
    f = tbl._lib.tb_patch_gn_stats
    assert f(ptrs, 4, 9, 1, 64, sp, 32, 16, None) == tbl.TB_ERR_DTYPE
    assert f(ptrs, 4, 2, 1, 60, sp, 32, 16, None) == tbl.TB_ERR_SHAPE        # C % G
    assert f(ptrs, 0, 2, 1, 64, sp, 32, 16, None) == tbl.TB_ERR_SHAPE        # P < 1
    assert f(ptrs, 4, 2, 1, 64, sp, 32, None, None) == tbl.TB_ERR_NULL       # partials
    assert f(ptrs, 4, 2, 1, 64, None, 32, 16, None) == tbl.TB_ERR_NULL       # spatial
    assert f(ptrs, 65, 2, 1, 64, (ctypes.c_int64 * 65)(*[1] * 65), 32, 16, None) == tbl.TB_ERR_UNSUPPORTED
    g = tbl._lib.tb_patch_gn_apply
    assert g(ptrs, ptrs, 4, 2, 1, 64, sp, 32, 16, None, None, ctypes.c_float(-1.0), 1, None) == tbl.TB_ERR_SHAPE
    assert g(ptrs, None, 4, 2, 1, 64, sp, 32, 16, None, None, ctypes.c_float(1e-6), 1, None) == tbl.TB_ERR_NULL
    assert g(ptrs, ptrs, 4, 2, 0, 64, sp, 32, 16, None, None, ctypes.c_float(1e-6), 1, None) == tbl.TB_OK


def test_status_strings(tbl):
    for s in range(7):
        assert tbl._lib.tb_status_string(s)
    assert tbl._lib.tb_status_string(99) == b"unknown status"


def test_ramp_stitch_rejects_bad_layouts_before_launch(tbl):
    def call(ay, ax, dtype=2):
        arr = (ctypes.c_void_p * 64)(*([16] * 64))
        a, b = ay.c(), ax.c()
        return tbl._lib.tb_stitch2d_ramp(arr, dtype, 1, 3, ctypes.byref(a), ctypes.byref(b), 16, None)
    good = tbl.RampAxis.spread(256, 64, 5, 8)
    assert good.origins == (0, 384, 768, 1152, 1536)
    assert call(good, good, dtype=5) == tbl.TB_ERR_DTYPE
    # last tile not ending at the canvas edge
    assert call(tbl.RampAxis((0, 384), 512, 1024, 32, 64), good) == tbl.TB_ERR_GEOMETRY
    # origins out of order
    assert call(tbl.RampAxis((0, 600, 512), 512, 1024, 32, 64), good) == tbl.TB_ERR_GEOMETRY
    # overlap shorter than the zero bands: the seam has no weight
    assert call(tbl.RampAxis((0, 500), 512, 1012, 32, 64), good) == tbl.TB_ERR_GEOMETRY
    # ramp of zero samples
    assert call(tbl.RampAxis((0, 384), 512, 896, 32, 0), good) == tbl.TB_ERR_GEOMETRY
    # four tiles with positive weight at one position
    dense = tbl.RampAxis(tuple(range(0, 97, 8)), 64, 160, 0, 1)
    assert call(dense, good) == tbl.TB_ERR_UNSUPPORTED
    # nothing to do
    arr = (ctypes.c_void_p * 64)()
    a, b = good.c(), good.c()
    assert tbl._lib.tb_stitch2d_ramp(arr, 2, 0, 3, ctypes.byref(a), ctypes.byref(b), None, None) == tbl.TB_OK


def test_patchify_layout_matches_the_oracle(tbl):
    from oracle.patchify import layout
    rnd = random.Random(11)
    for _ in range(2000):
        factor = rnd.choice([1, 2, 4, 8, 16])
        P = rnd.randint(1, tbl.TB_MAX_PATCHES)
        extent = factor * rnd.randint(0, 300)
        assert tbl.tb_patchify_layout(extent, factor, P) == tuple(map(list, layout(extent, factor, P)))


def test_patchify_layout_rejects_bad_counts(tbl):
    for args, st in (((209, 8, 3), tbl.TB_ERR_SHAPE), ((16, 0, 2), tbl.TB_ERR_SHAPE), ((16, 1, 0), tbl.TB_ERR_SHAPE),
                     ((-8, 8, 2), tbl.TB_ERR_SHAPE), ((64, 1, 65), tbl.TB_ERR_UNSUPPORTED)):
        with pytest.raises(tbl.TileBlendError) as e:
            tbl.tb_patchify_layout(*args)
        assert e.value.status == st


def test_patchify_and_gather_reject_before_launch(tbl):
    shape = (ctypes.c_int64 * 5)(1, 384, 13, 120, 208)
    ptrs = (ctypes.c_void_p * 3)(16, 32, 48)
    split = tbl._lib.tb_patchify
    assert split(16, 9, 5, shape, 4, 8, 3, 0, ptrs, None) == tbl.TB_ERR_DTYPE
    assert split(16, 2, 0, shape, 0, 8, 3, 0, ptrs, None) == tbl.TB_ERR_SHAPE       # ndim
    assert split(16, 2, 9, shape, 0, 8, 3, 0, ptrs, None) == tbl.TB_ERR_SHAPE       # ndim
    assert split(16, 2, 5, shape, 5, 8, 3, 0, ptrs, None) == tbl.TB_ERR_SHAPE       # axis
    assert split(16, 2, 5, shape, 4, 24, 3, 0, ptrs, None) == tbl.TB_ERR_SHAPE      # 208 is not whole bands of 24
    assert split(16, 2, 5, shape, 4, 8, 3, 71, ptrs, None) == tbl.TB_ERR_SHAPE      # slot < the largest band (72)
    assert split(16, 2, 5, shape, 4, 8, 3, -1, ptrs, None) == tbl.TB_ERR_SHAPE
    assert split(16, 2, 5, shape, 4, 8, 65, 0, ptrs, None) == tbl.TB_ERR_UNSUPPORTED
    assert split(None, 2, 5, shape, 4, 8, 3, 0, ptrs, None) == tbl.TB_ERR_NULL
    assert split(16, 2, 5, None, 4, 8, 3, 0, ptrs, None) == tbl.TB_ERR_NULL
    assert split(16, 2, 5, shape, 4, 8, 3, 0, None, None) == tbl.TB_ERR_NULL
    assert split(16, 2, 5, shape, 4, 8, 3, 0, (ctypes.c_void_p * 3)(16, None, 48), None) == tbl.TB_ERR_NULL
    neg = (ctypes.c_int64 * 5)(1, -384, 13, 120, 208)
    assert split(16, 2, 5, neg, 4, 8, 3, 0, ptrs, None) == tbl.TB_ERR_SHAPE
    # nothing to move: success without a launch, whatever the pointers
    empty = (ctypes.c_int64 * 5)(0, 384, 13, 120, 208)
    assert split(None, 2, 5, empty, 4, 8, 3, 0, (ctypes.c_void_p * 3)(), None) == tbl.TB_OK
    # more ranks than bands: the empty patches need no pointer (still no launch here)
    small = (ctypes.c_int64 * 2)(0, 16)
    assert split(None, 2, 2, small, 1, 8, 4, 0, (ctypes.c_void_p * 4)(), None) == tbl.TB_OK

    gather = tbl._lib.tb_gather_patches
    sizes = (ctypes.c_int64 * 3)(72, 72, 64)
    assert gather(ptrs, 3, (ctypes.c_int64 * 3)(72, 72, 63), 2, 5, shape, 4, 0, 16, None) == tbl.TB_ERR_SHAPE
    assert gather(ptrs, 3, (ctypes.c_int64 * 3)(72, -8, 144), 2, 5, shape, 4, 0, 16, None) == tbl.TB_ERR_SHAPE
    assert gather(ptrs, 3, None, 2, 5, shape, 4, 0, 16, None) == tbl.TB_ERR_NULL
    assert gather(ptrs, 0, sizes, 2, 5, shape, 4, 0, 16, None) == tbl.TB_ERR_SHAPE
    assert gather(ptrs, 3, sizes, 2, 5, shape, 4, 0, None, None) == tbl.TB_ERR_NULL
    assert gather(ptrs, 3, sizes, 2, 5, shape, 4, 70, 16, None) == tbl.TB_ERR_SHAPE
    assert gather(ptrs, 3, sizes, 7, 5, shape, 4, 0, 16, None) == tbl.TB_ERR_DTYPE
    # any sizes, not only whole bands, as long as they sum to the axis
    odd = (ctypes.c_int64 * 3)(1, 0, 207)
    assert gather((ctypes.c_void_p * 3)(16, None, 48), 3, odd, 2, 5, empty, 4, 0, 16, None) == tbl.TB_OK


def test_header_constants_match_the_binding(tbl):
    src = open(HEADER).read()
    for name in ("TB_MAX_TILES_PER_AXIS", "TB_MAX_TILES", "TB_GN_PARTS", "TB_NOALLOC_MAX_PARTIALS", "TB_MAX_PATCHES"):
        m = re.search(r"#define\s+%s\s+(\d+)" % name, src)
        assert m and int(m.group(1)) == getattr(tbl, name), name


def test_product_path_and_oracle_share_no_code():
    # the package never imports the oracle, and the oracle never imports the
    # package or links the library; only tests, the smoke check and the
    # benchmark's CPU legs bring the two together
    import ast
    import glob

    def imports(path):
        tree = ast.parse(open(path).read())
        names = set()
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                names.update(a.name.split(".")[0] for a in node.names)
            elif isinstance(node, ast.ImportFrom) and node.module:
                names.add(node.module.split(".")[0])
        return names

    for path in glob.glob(os.path.join(ROOT, "patch_groupnorm_gb300", "*.py")):
        assert "oracle" not in imports(path), path
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        assert "patch_groupnorm_gb300" not in imports(path), path
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.c")) + glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        assert "tileblend" not in open(path).read(), path
    for path in glob.glob(os.path.join(ROOT, "patch_groupnorm_gb300", "csrc", "*")):
        assert "oracle" not in open(path).read().lower(), path


# --------------------------------------------------------------------------
# row-sharded stitch layout and the gathered GroupNorm apply (host side)
# --------------------------------------------------------------------------

def _expected_shares(lay, world, planes, frames, width):
    """Tile rows dealt in rank order (the first ranks one more), each rank's
    output rows, and the bands crossing each rank boundary, recomputed from
    the oracle's geometry."""
    n = lay.n
    out = []
    begin = 0
    for r in range(world):
        rows = n // world + (1 if r < n % world else 0)
        end = begin + rows
        halo = lay.blends[begin] if (rows and begin > 0) else 0
        send = lay.blends[end] if (rows and end < n) else 0
        out.append((begin, end, sum(lay.kept[:begin]), sum(lay.kept[begin:end]), halo,
                    planes * frames * halo * width, planes * frames * send * width))
        begin = end
    return out


@pytest.mark.parametrize("case", [
    (None, (256, 64, 0.25, 8), (256, 64, 0.25, 8), 4, 3),
    (None, (200, 120, 0.25, 8), (256, 72, 0.25, 8), 1, 3),
    ((49, 16, 0.25, 1), (60, 32, 0.25, 8), (104, 32, 0.25, 8), 1, 3),
    (None, (30, 8, 0.0, 8), (20, 8, 0.0, 4), 2, 2),
])
def test_shard_layout_matches_the_oracle_geometry(tbl, case):
    at, ay, ax, B, C = case
    lt = axis_layout(*at) if at else None
    ly, lx = axis_layout(*ay), axis_layout(*ax)
    frames = sum(lt.extents) if lt else 1
    for world in (1, 2, 3, ly.n, ly.n + 3):
        want = _expected_shares(ly, world, B * C, frames, sum(lx.extents))
        for r in range(world):
            got = tbl.tb_stitch_shard_layout(tbl.Axis(*at) if at else None, tbl.Axis(*ay), tbl.Axis(*ax), B, C,
                                             world, r)
            assert (got.row_begin, got.row_end, got.out_row_begin, got.out_rows, got.halo_rows, got.halo_elems,
                    got.send_elems) == want[r], (world, r)
        # the shares tile the output rows exactly
        assert sum(w[3] for w in want) == ly.out_extent


@pytest.mark.parametrize("case", [
    ((49, 16, 0.25, 1), (60, 32, 0.25, 8), (104, 32, 0.25, 8), 1, 3),
    ((21, 8, 0.25, 1), (40, 16, 0.25, 4), (24, 16, 0.25, 4), 2, 2),
])
def test_frame_shard_layout_matches_the_oracle_geometry(tbl, case):
    at, ay, ax, B, C = case
    lt, ly, lx = axis_layout(*at), axis_layout(*ay), axis_layout(*ax)
    for world in (1, 2, 3, lt.n, lt.n + 3):
        # frame tiles dealt like rows; a band is e_t frames of every (i, j) tile
        want = _expected_shares(lt, world, B * C, 1, sum(ly.extents) * sum(lx.extents))
        for r in range(world):
            got = tbl.tb_stitch_shard_frames_layout(tbl.Axis(*at), tbl.Axis(*ay), tbl.Axis(*ax), B, C, world, r)
            assert (got.row_begin, got.row_end, got.out_row_begin, got.out_rows, got.halo_rows, got.halo_elems,
                    got.send_elems) == want[r], (world, r)


def test_shard_calls_reject_before_launch(tbl):
    ay, ax = tbl.Axis(256, 64, 0.25, 8), tbl.Axis(128, 64, 0.25, 8)
    a_y, a_x = ay.c(), ax.c()
    out = tbl.tb_shard_layout()
    f = tbl._lib.tb_stitch_shard_layout
    assert f(None, ctypes.byref(a_y), ctypes.byref(a_x), 1, 3, 0, 0, ctypes.byref(out)) == tbl.TB_ERR_SHAPE
    assert f(None, ctypes.byref(a_y), ctypes.byref(a_x), 1, 3, 2, 2, ctypes.byref(out)) == tbl.TB_ERR_SHAPE
    assert f(None, None, ctypes.byref(a_x), 1, 3, 2, 0, ctypes.byref(out)) == tbl.TB_ERR_NULL
    pack = tbl._lib.tb_stitch_halo_pack
    arr = (ctypes.c_void_p * 3)(16, 32, 48)
    # the last tile row lends no band; a row past the grid is refused
    assert pack(arr, 2, 1, 3, None, ctypes.byref(a_y), ctypes.byref(a_x), 5, 16, None) == tbl.TB_ERR_SHAPE
    assert pack(arr, 2, 1, 3, None, ctypes.byref(a_y), ctypes.byref(a_x), -1, 16, None) == tbl.TB_ERR_SHAPE
    assert pack(arr, 2, 1, 3, None, ctypes.byref(a_y), ctypes.byref(a_x), 0, None, None) == tbl.TB_ERR_NULL
    assert pack(arr, 9, 1, 3, None, ctypes.byref(a_y), ctypes.byref(a_x), 0, 16, None) == tbl.TB_ERR_DTYPE
    st = tbl._lib.tb_stitch2d_shard
    tiles = (ctypes.c_void_p * 9)(*([16] * 9))
    # rows 3..6 need the band of row 2
    assert st(tiles, None, 2, 1, 3, ctypes.byref(a_y), ctypes.byref(a_x), 3, 6, 16, 896, 1024, None) \
        == tbl.TB_ERR_NULL
    assert st(tiles, 16, 2, 1, 3, ctypes.byref(a_y), ctypes.byref(a_x), 3, 6, 16, 895, 1024, None) \
        == tbl.TB_ERR_SHAPE
    assert st(tiles, 16, 2, 1, 3, ctypes.byref(a_y), ctypes.byref(a_x), 4, 3, 16, 0, 1024, None) \
        == tbl.TB_ERR_SHAPE
    assert st(tiles, 16, 2, 1, 3, ctypes.byref(a_y), ctypes.byref(a_x), 0, 7, 16, 0, 1024, None) \
        == tbl.TB_ERR_SHAPE
    # an empty share writes nothing
    assert st(None, None, 2, 1, 3, ctypes.byref(a_y), ctypes.byref(a_x), 6, 6, None, 0, 1024, None) == tbl.TB_OK
    # the frame forms need the frame axis
    f = tbl._lib.tb_stitch_shard_frames_layout
    assert f(None, ctypes.byref(a_y), ctypes.byref(a_x), 1, 3, 2, 0, ctypes.byref(out)) == tbl.TB_ERR_NULL
    pf = tbl._lib.tb_stitch_halo_pack_frames
    assert pf(arr, 2, 1, 3, None, ctypes.byref(a_y), ctypes.byref(a_x), 0, 16, None) == tbl.TB_ERR_NULL
    a_t = tbl.Axis(49, 16, 0.25, 1).c()
    assert pf(arr, 2, 1, 3, ctypes.byref(a_t), ctypes.byref(a_y), ctypes.byref(a_x), 4, 16, None) == tbl.TB_ERR_SHAPE
    sf = tbl._lib.tb_stitch3d_shard_frames
    # frame tiles 2..5 need the band of frame tile 1
    assert sf(tiles, None, 2, 1, 3, ctypes.byref(a_t), ctypes.byref(a_y), ctypes.byref(a_x), 2, 5, 16, 25, 1536,
              1024, None) == tbl.TB_ERR_NULL


def test_gathered_apply_rejects_before_launch(tbl):
    ptrs = (ctypes.c_void_p * 1)(16)
    sp = (ctypes.c_int64 * 1)(100)
    g = tbl._lib.tb_patch_gn_apply_gathered
    eps = ctypes.c_float(1e-6)
    assert g(ptrs, ptrs, 1, 2, 1, 64, sp, 32, 16, 0, None, None, eps, 1, None) == tbl.TB_ERR_SHAPE      # R < 1
    assert g(ptrs, ptrs, 1, 2, 1, 64, sp, 32, 16, 65537, None, None, eps, 1, None) == tbl.TB_ERR_UNSUPPORTED
    assert g(ptrs, ptrs, 1, 2, 1, 64, sp, 32, None, 4, None, None, eps, 1, None) == tbl.TB_ERR_NULL
    assert g(ptrs, ptrs, 1, 2, 1, 60, sp, 32, 16, 4, None, None, eps, 1, None) == tbl.TB_ERR_SHAPE     # C % G


def test_ramp_spread_matches_the_oracle_on_every_tile():
    # the library's planner spread against the oracle's, interior tiles included
    import random
    from oracle.ramp import evenly_spread_origins
    from patch_groupnorm_gb300 import build
    build.build()
    from patch_groupnorm_gb300 import tileblend as tbl
    rnd = random.Random(5)
    checked = 0
    for _ in range(500):
        tile = rnd.randint(2, 80)
        ext = rnd.randint(tile, 10 * tile)
        n = 1 if ext == tile else rnd.randint(2, 20)
        if n > 1 and -(-(ext - tile) // (n - 1)) > tile:
            continue                                   # would leave a gap: refused, checked below
        scale = rnd.choice([1, 2, 8, 16])
        got = tbl.RampAxis.spread(ext, tile, n, scale)
        assert list(got.origins) == evenly_spread_origins(ext, tile, n, scale)
        assert (got.tile_extent, got.out_extent, got.zero, got.ramp) == (tile * scale, ext * scale, 4 * scale,
                                                                         8 * scale)
        checked += 1
    assert checked > 300


def test_ramp_spread_rejects_bad_layouts(tbl):
    org = (ctypes.c_int64 * 64)()
    a = tbl.tb_ramp_axis()
    f = tbl._lib.tb_ramp_axis_spread
    assert f(100, 32, 0, 8, 4, 8, org, ctypes.byref(a)) == tbl.TB_ERR_GEOMETRY      # no tiles
    assert f(100, 32, 1, 8, 4, 8, org, ctypes.byref(a)) == tbl.TB_ERR_GEOMETRY      # one tile, not the canvas
    assert f(100, 32, 2, 8, 4, 8, org, ctypes.byref(a)) == tbl.TB_ERR_GEOMETRY      # a 36-latent gap
    assert f(100, 132, 4, 8, 4, 8, org, ctypes.byref(a)) == tbl.TB_ERR_GEOMETRY     # tile past the canvas
    assert f(100, 32, 4, 8, 4, 0, org, ctypes.byref(a)) == tbl.TB_ERR_GEOMETRY      # no ramp
    assert f(10000, 32, 65, 8, 4, 8, org, ctypes.byref(a)) == tbl.TB_ERR_UNSUPPORTED
    assert f(100, 32, 4, 8, 4, 8, None, ctypes.byref(a)) == tbl.TB_ERR_NULL
    assert f(100, 32, 4, 8, 4, 8, org, ctypes.byref(a)) == tbl.TB_OK
    assert list(org[:4]) == [0, 22 * 8, 45 * 8, 68 * 8] and a.n_tiles == 4
