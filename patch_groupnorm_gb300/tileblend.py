"""Python binding of libtileblend (include/tileblend.h).

Argument marshalling only: every step of the stitch and of PatchGroupNorm
runs in the library's CUDA kernels.  Tensors must be CUDA tensors on the
current device, contiguous, of one dtype (float32, float16 or bfloat16).
Calls are asynchronous on the current torch stream unless ``stream`` (a
``torch.cuda.Stream`` or a raw ``cudaStream_t`` integer) is given.

There is no fallback: if the compiled library is missing, importing this
module raises.
"""
import ctypes
import functools
import os
from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# TILEBLEND_LIB selects another build of the same library (a variant built by
# build.build(variant=...), e.g. with in-kernel bounds checks).
LIB_PATH = os.environ.get("TILEBLEND_LIB") or os.path.join(_HERE, "_build", "libtileblend.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libtileblend.so is not built (expected at %s); run "
        "`python -c 'import __graft_entry__ as g; g.build()'` or "
        "`python patch_groupnorm_gb300/build.py`" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

# ---------------------------------------------------------------------------
# C declarations
# ---------------------------------------------------------------------------

TB_OK, TB_ERR_NULL, TB_ERR_DTYPE, TB_ERR_SHAPE, TB_ERR_GEOMETRY, TB_ERR_UNSUPPORTED, TB_ERR_CUDA = range(7)
TB_F32, TB_F16, TB_BF16 = 0, 1, 2
TB_MAX_TILES_PER_AXIS = 64
TB_MAX_TILES = 1024
TB_GN_PARTS = 8

_DTYPES = {torch.float32: TB_F32, torch.float16: TB_F16, torch.bfloat16: TB_BF16}


class tb_axis(ctypes.Structure):
    _fields_ = [("latent_extent", ctypes.c_int32), ("latent_tile", ctypes.c_int32), ("overlap", ctypes.c_double),
                ("scale", ctypes.c_int32), ("blend_extent", ctypes.c_int32), ("row_limit", ctypes.c_int32)]


class tb_ramp_axis(ctypes.Structure):
    _fields_ = [("n_tiles", ctypes.c_int32), ("tile_extent", ctypes.c_int32), ("out_extent", ctypes.c_int32),
                ("zero", ctypes.c_int32), ("ramp", ctypes.c_int32), ("origins", ctypes.POINTER(ctypes.c_int64))]


class tb_gn_partial(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("mean", ctypes.c_float), ("m2", ctypes.c_float)]


class tb_shard_layout(ctypes.Structure):
    _fields_ = [("row_begin", ctypes.c_int32), ("row_end", ctypes.c_int32), ("out_row_begin", ctypes.c_int64),
                ("out_rows", ctypes.c_int64), ("halo_rows", ctypes.c_int32), ("halo_elems", ctypes.c_int64),
                ("send_elems", ctypes.c_int64)]


_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
_P_vp = ctypes.POINTER(ctypes.c_void_p)
_P_i32 = ctypes.POINTER(ctypes.c_int32)
_P_i64 = ctypes.POINTER(ctypes.c_int64)
_P_axis = ctypes.POINTER(tb_axis)

_lib.tb_version.restype = ctypes.c_size_t
_lib.tb_version.argtypes = []
_lib.tb_status_string.restype = ctypes.c_char_p
_lib.tb_status_string.argtypes = [ctypes.c_int]
_lib.tb_last_cuda_error.restype = ctypes.c_int
_lib.tb_last_cuda_error.argtypes = []
_lib.tb_axis_layout.restype = ctypes.c_int
_lib.tb_axis_layout.argtypes = [_P_axis, _i32, _P_i32, _P_i64, _P_i32, _P_i32, _P_i32, _P_i64]
_lib.tb_stitch2d.restype = ctypes.c_int
_lib.tb_stitch2d.argtypes = [_P_vp, ctypes.c_int, _i64, _i64, _P_axis, _P_axis, _vp, _i64, _i64, _vp]
_lib.tb_stitch3d.restype = ctypes.c_int
_lib.tb_stitch3d.argtypes = [_P_vp, ctypes.c_int, _i64, _i64, _P_axis, _P_axis, _P_axis, _vp, _i64, _i64, _i64, _vp]
_lib.tb_patch_gn_stats.restype = ctypes.c_int
_lib.tb_patch_gn_stats.argtypes = [_P_vp, _i32, ctypes.c_int, _i64, _i64, _P_i64, _i32, _vp, _vp]
_lib.tb_patch_gn_apply.restype = ctypes.c_int
_lib.tb_patch_gn_apply.argtypes = [_P_vp, _P_vp, _i32, ctypes.c_int, _i64, _i64, _P_i64, _i32, _vp, _vp, _vp,
                                   ctypes.c_float, _i32, _vp]

_lib.tb_patch_gn_apply_gathered.restype = ctypes.c_int
_lib.tb_patch_gn_apply_gathered.argtypes = [_P_vp, _P_vp, _i32, ctypes.c_int, _i64, _i64, _P_i64, _i32, _vp, _i32,
                                            _vp, _vp, ctypes.c_float, _i32, _vp]
_lib.tb_stitch_shard_layout.restype = ctypes.c_int
_lib.tb_stitch_shard_layout.argtypes = [_P_axis, _P_axis, _P_axis, _i64, _i64, _i32, _i32,
                                        ctypes.POINTER(tb_shard_layout)]
_lib.tb_stitch_halo_pack.restype = ctypes.c_int
_lib.tb_stitch_halo_pack.argtypes = [_P_vp, ctypes.c_int, _i64, _i64, _P_axis, _P_axis, _P_axis, _i32, _vp, _vp]
_lib.tb_stitch2d_shard.restype = ctypes.c_int
_lib.tb_stitch2d_shard.argtypes = [_P_vp, _vp, ctypes.c_int, _i64, _i64, _P_axis, _P_axis, _i32, _i32, _vp, _i64,
                                   _i64, _vp]
_lib.tb_stitch_shard_frames_layout.restype = ctypes.c_int
_lib.tb_stitch_shard_frames_layout.argtypes = [_P_axis, _P_axis, _P_axis, _i64, _i64, _i32, _i32,
                                               ctypes.POINTER(tb_shard_layout)]
_lib.tb_stitch_halo_pack_frames.restype = ctypes.c_int
_lib.tb_stitch_halo_pack_frames.argtypes = [_P_vp, ctypes.c_int, _i64, _i64, _P_axis, _P_axis, _P_axis, _i32, _vp,
                                            _vp]
_lib.tb_stitch3d_shard_frames.restype = ctypes.c_int
_lib.tb_stitch3d_shard_frames.argtypes = [_P_vp, _vp, ctypes.c_int, _i64, _i64, _P_axis, _P_axis, _P_axis, _i32,
                                          _i32, _vp, _i64, _i64, _i64, _vp]
_lib.tb_stitch3d_shard.restype = ctypes.c_int
_lib.tb_stitch3d_shard.argtypes = [_P_vp, _vp, ctypes.c_int, _i64, _i64, _P_axis, _P_axis, _P_axis, _i32, _i32, _vp,
                                   _i64, _i64, _i64, _vp]

_lib.tb_device_status.restype = ctypes.c_int
_lib.tb_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), _i32]
TB_DEV_OK, TB_DEV_WAIT_TIMEOUT, TB_DEV_OUT_OF_BOUNDS = 0, 1, 2

_lib.tb_ramp_axis_spread.restype = ctypes.c_int
_lib.tb_ramp_axis_spread.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _P_i64, ctypes.POINTER(tb_ramp_axis)]
_lib.tb_stitch2d_ramp.restype = ctypes.c_int
_lib.tb_stitch2d_ramp.argtypes = [_P_vp, ctypes.c_int, _i64, _i64, ctypes.POINTER(tb_ramp_axis),
                                  ctypes.POINTER(tb_ramp_axis), _vp, _vp]
_lib.tb_patch_group_norm_noalloc.restype = ctypes.c_int
_lib.tb_patch_group_norm_noalloc.argtypes = [_P_vp, _P_vp, _i32, ctypes.c_int, _i64, _i64, _P_i64, _i32, _vp, _vp,
                                             ctypes.c_float, _i32, _vp]
TB_NOALLOC_MAX_PARTIALS = 65536
_lib.tb_patchify_layout.restype = ctypes.c_int
_lib.tb_patchify_layout.argtypes = [_i64, _i32, _i32, _P_i64, _P_i64]
_lib.tb_patchify.restype = ctypes.c_int
_lib.tb_patchify.argtypes = [_vp, ctypes.c_int, _i32, _P_i64, _i32, _i32, _i32, _i64, _P_vp, _vp]
_lib.tb_gather_patches.restype = ctypes.c_int
_lib.tb_gather_patches.argtypes = [_P_vp, _i32, _P_i64, ctypes.c_int, _i32, _P_i64, _i32, _i64, _vp, _vp]
TB_MAX_PATCHES = 64

EXPORTED = ("tb_version", "tb_status_string", "tb_last_cuda_error", "tb_axis_layout", "tb_stitch2d",
            "tb_stitch3d", "tb_stitch_shard_layout", "tb_stitch_halo_pack", "tb_stitch2d_shard",
            "tb_stitch3d_shard", "tb_stitch2d_ramp", "tb_patch_gn_stats", "tb_patch_gn_apply",
            "tb_patch_gn_apply_gathered", "tb_patch_group_norm_noalloc", "tb_patchify_layout", "tb_patchify",
            "tb_gather_patches", "tb_device_status", "tb_ramp_axis_spread", "tb_stitch_shard_frames_layout",
            "tb_stitch_halo_pack_frames", "tb_stitch3d_shard_frames")


class TileBlendError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = "%s: %s" % (where, _lib.tb_status_string(status).decode())
        if status == TB_ERR_CUDA:
            msg += " (cudaError %d)" % _lib.tb_last_cuda_error()
        super().__init__(msg)
        self.status = status


def _check(status: int, where: str) -> None:
    if status != TB_OK:
        raise TileBlendError(status, where)


def tb_version() -> int:
    return int(_lib.tb_version())


def tb_device_status(clear: bool = False) -> int:
    """The device status word (0 = no kernel reported a problem); synchronises."""
    v = ctypes.c_uint32(0)
    _check(_lib.tb_device_status(ctypes.byref(v), 1 if clear else 0), "tb_device_status")
    return int(v.value)


# ---------------------------------------------------------------------------
# geometry
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Axis:
    """Tile-grid parameters of one axis (see tb_axis in tileblend.h)."""
    latent_extent: int
    latent_tile: int
    overlap: float
    scale: int
    blend_extent: int = -1   # < 0: stock value
    row_limit: int = 0       # <= 0: stock value

    def c(self) -> tb_axis:
        return tb_axis(self.latent_extent, self.latent_tile, float(self.overlap), self.scale,
                       self.blend_extent, self.row_limit)


@dataclass(frozen=True)
class Layout:
    n: int
    origins: List[int]     # in decoded samples
    extents: List[int]
    blends: List[int]
    kept: List[int]
    out_extent: int


@functools.lru_cache(maxsize=256)
def tb_axis_layout(axis: Axis) -> Layout:
    """The library's derived geometry of one axis (host only; cached per
    parameter set)."""
    a = axis.c()
    n = ctypes.c_int32(0)
    cap = TB_MAX_TILES_PER_AXIS
    org = (ctypes.c_int64 * cap)()
    ext, bl, kp = (ctypes.c_int32 * cap)(), (ctypes.c_int32 * cap)(), (ctypes.c_int32 * cap)()
    out = ctypes.c_int64(0)
    _check(_lib.tb_axis_layout(ctypes.byref(a), cap, ctypes.byref(n), org, ext, bl, kp, ctypes.byref(out)),
           "tb_axis_layout")
    k = n.value
    return Layout(k, list(org[:k]), list(ext[:k]), list(bl[:k]), list(kp[:k]), out.value)


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError("unsupported dtype %s" % t.dtype)
    return _DTYPES[t.dtype]


def _cuda_contig(t: torch.Tensor, what: str) -> None:
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)


def _ptr_array(ptrs: Sequence[int]):
    return (ctypes.c_void_p * max(1, len(ptrs)))(*ptrs)


# ---------------------------------------------------------------------------
# stitch
# ---------------------------------------------------------------------------

def tb_stitch2d(tiles: Sequence[Sequence[torch.Tensor]], ay: Axis, ax: Axis, out: torch.Tensor, stream=None) -> torch.Tensor:
    """Stitch ``tiles[i][j]`` ([B, C, L_y(i), L_x(j)]) into ``out`` ([B, C, H, W])."""
    _cuda_contig(out, "out")
    B, C, H, W = out.shape
    ly, lx = tb_axis_layout(ay), tb_axis_layout(ax)
    ptrs = []
    if len(tiles) != ly.n:
        raise ValueError("expected %d tile rows, got %d" % (ly.n, len(tiles)))
    dt = out.dtype
    for i, row in enumerate(tiles):
        if len(row) != lx.n:
            raise ValueError("expected %d tiles in row %d, got %d" % (lx.n, i, len(row)))
        Ly = ly.extents[i]
        for j, t in enumerate(row):
            if t.dtype != dt or t.shape != (B, C, Ly, lx.extents[j]) or not t.is_cuda or not t.is_contiguous():
                _cuda_contig(t, "tile (%d,%d)" % (i, j))
                raise ValueError("tile (%d,%d) has %s %s, expected %s %s" % (
                    i, j, t.dtype, tuple(t.shape), dt, (B, C, Ly, lx.extents[j])))
            ptrs.append(t.data_ptr())
    a_y, a_x = ay.c(), ax.c()
    _check(_lib.tb_stitch2d(_ptr_array(ptrs), _dtype_code(out), B, C, ctypes.byref(a_y), ctypes.byref(a_x),
                            out.data_ptr(), H, W, _stream_handle(stream)), "tb_stitch2d")
    return out


def tb_stitch3d(tiles, at: Axis, ay: Axis, ax: Axis, out: torch.Tensor, stream=None) -> torch.Tensor:
    """Stitch ``tiles[k][i][j]`` ([B, C, L_t(k), L_y(i), L_x(j)]) into ``out``
    ([B, C, T, H, W])."""
    _cuda_contig(out, "out")
    B, C, T, H, W = out.shape
    lt, ly, lx = tb_axis_layout(at), tb_axis_layout(ay), tb_axis_layout(ax)
    ptrs = []
    if len(tiles) != lt.n:
        raise ValueError("expected %d frame tiles, got %d" % (lt.n, len(tiles)))
    for k, plane in enumerate(tiles):
        if len(plane) != ly.n:
            raise ValueError("expected %d tile rows" % ly.n)
        for i, row in enumerate(plane):
            if len(row) != lx.n:
                raise ValueError("expected %d tiles per row" % lx.n)
            for j, t in enumerate(row):
                _cuda_contig(t, "tile (%d,%d,%d)" % (k, i, j))
                exp = (B, C, lt.extents[k], ly.extents[i], lx.extents[j])
                if t.dtype != out.dtype or tuple(t.shape) != exp:
                    raise ValueError("tile (%d,%d,%d) has %s %s, expected %s %s" % (
                        k, i, j, t.dtype, tuple(t.shape), out.dtype, exp))
                ptrs.append(t.data_ptr())
    a_t, a_y, a_x = at.c(), ay.c(), ax.c()
    _check(_lib.tb_stitch3d(_ptr_array(ptrs), _dtype_code(out), B, C, ctypes.byref(a_t), ctypes.byref(a_y),
                            ctypes.byref(a_x), out.data_ptr(), T, H, W, _stream_handle(stream)), "tb_stitch3d")
    return out


def tb_stitch2d_raw(tile_ptrs: Sequence[int], dtype: int, B: int, C: int, ay: Axis, ax: Axis, out_ptr: int,
                    H: int, W: int, stream=None) -> None:
    """Pointer-level call (no tensor checks), for timing the bare C ABI."""
    a_y, a_x = ay.c(), ax.c()
    _check(_lib.tb_stitch2d(_ptr_array(tile_ptrs), dtype, B, C, ctypes.byref(a_y), ctypes.byref(a_x), out_ptr,
                            H, W, _stream_handle(stream)), "tb_stitch2d")


# ---------------------------------------------------------------------------
# row-sharded stitch
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class ShardLayout:
    row_begin: int
    row_end: int
    out_row_begin: int
    out_rows: int
    halo_rows: int
    halo_elems: int
    send_elems: int


def _axis_ref(a: Optional[Axis]):
    if a is None:
        return None, None
    c = a.c()
    return c, ctypes.byref(c)


def tb_stitch_shard_layout(at: Optional[Axis], ay: Axis, ax: Axis, B: int, C: int, world: int,
                           rank: int) -> ShardLayout:
    """Rank ``rank``'s share of a stitch whose tile rows are split over
    ``world`` ranks (host only)."""
    _, pt = _axis_ref(at)
    _, py = _axis_ref(ay)
    _, px = _axis_ref(ax)
    out = tb_shard_layout()
    _check(_lib.tb_stitch_shard_layout(pt, py, px, B, C, world, rank, ctypes.byref(out)), "tb_stitch_shard_layout")
    return ShardLayout(out.row_begin, out.row_end, out.out_row_begin, out.out_rows, out.halo_rows, out.halo_elems,
                       out.send_elems)


def _flat_tiles(tiles, ndim: int) -> List[torch.Tensor]:
    if ndim == 2:
        return [t for row in tiles for t in row]
    return [t for plane in tiles for row in plane for t in row]


def tb_stitch_halo_pack(row_tiles, at: Optional[Axis], ay: Axis, ax: Axis, row: int, halo: torch.Tensor,
                        stream=None) -> torch.Tensor:
    """Pack the last e_y(row + 1) rows of every tile of tile row ``row`` into
    ``halo`` (1D, ``send_elems`` elements).  ``row_tiles`` is the list of the
    row's tiles: ``[t_j]`` for a 2D grid, ``[[t_kj]]`` (frame tile major) for
    a 3D grid."""
    flat = list(row_tiles) if at is None else [t for per_k in row_tiles for t in per_k]
    for q, t in enumerate(flat):
        _cuda_contig(t, "tile %d" % q)
    _cuda_contig(halo, "halo")
    B, C = flat[0].shape[:2]
    _, pt = _axis_ref(at)
    _, py = _axis_ref(ay)
    _, px = _axis_ref(ax)
    _check(_lib.tb_stitch_halo_pack(_ptr_array([t.data_ptr() for t in flat]), _dtype_code(halo), B, C, pt, py, px,
                                    row, halo.data_ptr(), _stream_handle(stream)), "tb_stitch_halo_pack")
    return halo


def tb_stitch2d_shard(tiles, halo: Optional[torch.Tensor], ay: Axis, ax: Axis, row_begin: int, row_end: int,
                      out: torch.Tensor, stream=None) -> torch.Tensor:
    """Stitch tile rows [row_begin, row_end) (``tiles[i - row_begin][j]``)
    with the band ``halo`` of the row above into ``out`` ([B, C, out_rows,
    W])."""
    _cuda_contig(out, "out")
    B, C, H, W = out.shape
    flat = _flat_tiles(tiles, 2)
    for q, t in enumerate(flat):
        _cuda_contig(t, "tile %d" % q)
        if t.dtype != out.dtype:
            raise ValueError("tile %d has dtype %s, out %s" % (q, t.dtype, out.dtype))
    hp = None
    if halo is not None:
        _cuda_contig(halo, "halo")
        hp = halo.data_ptr()
    a_y, a_x = ay.c(), ax.c()
    _check(_lib.tb_stitch2d_shard(_ptr_array([t.data_ptr() for t in flat]), hp, _dtype_code(out), B, C,
                                  ctypes.byref(a_y), ctypes.byref(a_x), row_begin, row_end, out.data_ptr(), H, W,
                                  _stream_handle(stream)), "tb_stitch2d_shard")
    return out


def tb_stitch3d_shard(tiles, halo: Optional[torch.Tensor], at: Axis, ay: Axis, ax: Axis, row_begin: int,
                      row_end: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    """3D form of ``tb_stitch2d_shard``: ``tiles[k][i - row_begin][j]``,
    ``out`` [B, C, T, out_rows, W]."""
    _cuda_contig(out, "out")
    B, C, T, H, W = out.shape
    flat = _flat_tiles(tiles, 3)
    for q, t in enumerate(flat):
        _cuda_contig(t, "tile %d" % q)
        if t.dtype != out.dtype:
            raise ValueError("tile %d has dtype %s, out %s" % (q, t.dtype, out.dtype))
    hp = None
    if halo is not None:
        _cuda_contig(halo, "halo")
        hp = halo.data_ptr()
    a_t, a_y, a_x = at.c(), ay.c(), ax.c()
    _check(_lib.tb_stitch3d_shard(_ptr_array([t.data_ptr() for t in flat]), hp, _dtype_code(out), B, C,
                                  ctypes.byref(a_t), ctypes.byref(a_y), ctypes.byref(a_x), row_begin, row_end,
                                  out.data_ptr(), T, H, W, _stream_handle(stream)), "tb_stitch3d_shard")
    return out


def tb_stitch_shard_frames_layout(at: Axis, ay: Axis, ax: Axis, B: int, C: int, world: int,
                                  rank: int) -> ShardLayout:
    """Rank ``rank``'s share of a video stitch whose frame tiles are split
    over ``world`` ranks (host only; the fields count frame tiles and output
    frames)."""
    a_t, a_y, a_x = at.c(), ay.c(), ax.c()
    out = tb_shard_layout()
    _check(_lib.tb_stitch_shard_frames_layout(ctypes.byref(a_t), ctypes.byref(a_y), ctypes.byref(a_x), B, C, world,
                                              rank, ctypes.byref(out)), "tb_stitch_shard_frames_layout")
    return ShardLayout(out.row_begin, out.row_end, out.out_row_begin, out.out_rows, out.halo_rows, out.halo_elems,
                       out.send_elems)


def tb_stitch_halo_pack_frames(frame_tiles, at: Axis, ay: Axis, ax: Axis, frame_tile: int, halo: torch.Tensor,
                               stream=None) -> torch.Tensor:
    """Pack the last e_t(frame_tile + 1) frames of every tile of frame tile
    ``frame_tile`` (``frame_tiles[i][j]``) into ``halo``."""
    flat = [t for row in frame_tiles for t in row]
    for q, t in enumerate(flat):
        _cuda_contig(t, "tile %d" % q)
    _cuda_contig(halo, "halo")
    B, C = flat[0].shape[:2]
    a_t, a_y, a_x = at.c(), ay.c(), ax.c()
    _check(_lib.tb_stitch_halo_pack_frames(_ptr_array([t.data_ptr() for t in flat]), _dtype_code(halo), B, C,
                                           ctypes.byref(a_t), ctypes.byref(a_y), ctypes.byref(a_x), frame_tile,
                                           halo.data_ptr(), _stream_handle(stream)), "tb_stitch_halo_pack_frames")
    return halo


def tb_stitch3d_shard_frames(tiles, halo: Optional[torch.Tensor], at: Axis, ay: Axis, ax: Axis, frame_begin: int,
                             frame_end: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    """Stitch frame tiles [frame_begin, frame_end) (``tiles[k - frame_begin][i][j]``)
    with the band ``halo`` of the frame tile before into ``out``
    ([B, C, out_frames, H, W])."""
    _cuda_contig(out, "out")
    B, C, T, H, W = out.shape
    flat = _flat_tiles(tiles, 3)
    for q, t in enumerate(flat):
        _cuda_contig(t, "tile %d" % q)
        if t.dtype != out.dtype:
            raise ValueError("tile %d has dtype %s, out %s" % (q, t.dtype, out.dtype))
    hp = None
    if halo is not None:
        _cuda_contig(halo, "halo")
        hp = halo.data_ptr()
    a_t, a_y, a_x = at.c(), ay.c(), ax.c()
    _check(_lib.tb_stitch3d_shard_frames(_ptr_array([t.data_ptr() for t in flat]), hp, _dtype_code(out), B, C,
                                         ctypes.byref(a_t), ctypes.byref(a_y), ctypes.byref(a_x), frame_begin,
                                         frame_end, out.data_ptr(), T, H, W, _stream_handle(stream)),
           "tb_stitch3d_shard_frames")
    return out


# ---------------------------------------------------------------------------
# normalised-ramp stitch
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class RampAxis:
    """One axis of a normalised-ramp tile layout (see tb_ramp_axis)."""
    origins: Tuple[int, ...]   # output samples, ascending, first 0, last + tile_extent == out_extent
    tile_extent: int
    out_extent: int
    zero: int                  # samples of zero weight next to a shared edge
    ramp: int                  # samples over which the weight rises to 1

    @staticmethod
    def spread(latent_extent: int, latent_tile: int, n_tiles: int, scale: int, zero_latents: int = 4,
               ramp_latents: int = 8) -> "RampAxis":
        """The library's layout of n_tiles tiles spread edge to edge
        (tb_ramp_axis_spread)."""
        org = (ctypes.c_int64 * max(1, n_tiles))()
        a = tb_ramp_axis()
        _check(_lib.tb_ramp_axis_spread(latent_extent, latent_tile, n_tiles, scale, zero_latents, ramp_latents, org,
                                        ctypes.byref(a)), "tb_ramp_axis_spread")
        return RampAxis(tuple(org[:n_tiles]), a.tile_extent, a.out_extent, a.zero, a.ramp)

    def c(self):
        arr = (ctypes.c_int64 * len(self.origins))(*self.origins)
        st = tb_ramp_axis(len(self.origins), self.tile_extent, self.out_extent, self.zero, self.ramp,
                          ctypes.cast(arr, ctypes.POINTER(ctypes.c_int64)))
        st._keep = arr  # the struct points into this array
        return st


def tb_stitch2d_ramp(tiles: Sequence[Sequence[torch.Tensor]], ay: RampAxis, ax: RampAxis, out: torch.Tensor,
                     stream=None) -> torch.Tensor:
    """Normalised-ramp stitch of ``tiles[i][j]`` ([B, C, ay.tile_extent,
    ax.tile_extent]) into ``out`` ([B, C, ay.out_extent, ax.out_extent])."""
    _cuda_contig(out, "out")
    B, C, H, W = out.shape
    if (H, W) != (ay.out_extent, ax.out_extent):
        raise ValueError("out must be [B, C, %d, %d]" % (ay.out_extent, ax.out_extent))
    if len(tiles) != len(ay.origins) or any(len(r) != len(ax.origins) for r in tiles):
        raise ValueError("expected a %d x %d tile grid" % (len(ay.origins), len(ax.origins)))
    shape = (B, C, ay.tile_extent, ax.tile_extent)
    ptrs = []
    for i, row in enumerate(tiles):
        for j, t in enumerate(row):
            if t.dtype != out.dtype or t.shape != shape or not t.is_cuda or not t.is_contiguous():
                _cuda_contig(t, "tile (%d,%d)" % (i, j))
                raise ValueError("tile (%d,%d) has %s %s, expected %s %s" % (i, j, t.dtype, tuple(t.shape),
                                                                            out.dtype, shape))
            ptrs.append(t.data_ptr())
    a_y, a_x = ay.c(), ax.c()
    _check(_lib.tb_stitch2d_ramp(_ptr_array(ptrs), _dtype_code(out), B, C, ctypes.byref(a_y), ctypes.byref(a_x),
                                 out.data_ptr(), _stream_handle(stream)), "tb_stitch2d_ramp")
    return out


# ---------------------------------------------------------------------------
# PatchGroupNorm
# ---------------------------------------------------------------------------

def _gn_args(patches: Sequence[torch.Tensor]) -> Tuple[int, int, int, list, list]:
    if len(patches) == 0:
        raise ValueError("at least one patch")
    N, C = patches[0].shape[:2]
    spatial = []
    ptrs = []
    for q, t in enumerate(patches):
        _cuda_contig(t, "patch %d" % q)
        if t.dtype != patches[0].dtype or tuple(t.shape[:2]) != (N, C):
            raise ValueError("patch %d: dtype/leading dims differ from patch 0" % q)
        s = 1
        for d in t.shape[2:]:
            s *= d
        spatial.append(s)
        ptrs.append(t.data_ptr())
    return N, C, _dtype_code(patches[0]), spatial, ptrs


def new_partials(P: int, N: int, G: int, device=None) -> torch.Tensor:
    """Device buffer for the P * N * G * TB_GN_PARTS tb_gn_partial records
    (16 bytes each) that tb_patch_gn_stats writes."""
    return torch.empty((P, N, G, TB_GN_PARTS, 2), dtype=torch.int64, device=device or torch.device("cuda"))


def tb_patch_gn_stats(patches: Sequence[torch.Tensor], G: int, partials: torch.Tensor, stream=None) -> torch.Tensor:
    """(count, mean, M2) of every part of every (patch, sample, group) into
    ``partials`` (a [P, N, G, TB_GN_PARTS, 2] int64 buffer from
    ``new_partials``)."""
    N, C, dt, spatial, ptrs = _gn_args(patches)
    P = len(patches)
    _cuda_contig(partials, "partials")
    if partials.numel() * partials.element_size() != P * N * G * TB_GN_PARTS * 16:
        raise ValueError("partials must hold P*N*G*TB_GN_PARTS 16-byte records")
    sp = (ctypes.c_int64 * P)(*spatial)
    _check(_lib.tb_patch_gn_stats(_ptr_array(ptrs), P, dt, N, C, sp, G, partials.data_ptr(), _stream_handle(stream)),
           "tb_patch_gn_stats")
    return partials


def tb_patch_gn_apply(patches: Sequence[torch.Tensor], outs: Sequence[torch.Tensor], G: int, partials: torch.Tensor,
                      gamma: Optional[torch.Tensor], beta: Optional[torch.Tensor], eps: float, silu: bool = True,
                      stream=None) -> Sequence[torch.Tensor]:
    """Normalise every patch with the pooled statistics of ``partials``;
    ``outs[p]`` may be ``patches[p]``."""
    N, C, dt, spatial, ptrs = _gn_args(patches)
    P = len(patches)
    if len(outs) != P:
        raise ValueError("one output per patch")
    optrs = []
    for q, (o, t) in enumerate(zip(outs, patches)):
        _cuda_contig(o, "out %d" % q)
        if o.shape != t.shape or o.dtype != t.dtype:
            raise ValueError("out %d must match patch %d" % (q, q))
        optrs.append(o.data_ptr())
    for name, v in (("gamma", gamma), ("beta", beta)):
        if v is not None:
            _cuda_contig(v, name)
            if v.numel() != C or v.dtype != patches[0].dtype:
                raise ValueError("%s must be [C] of the patches' dtype" % name)
    _cuda_contig(partials, "partials")
    if partials.numel() * partials.element_size() != P * N * G * TB_GN_PARTS * 16:
        raise ValueError("partials must hold P*N*G*TB_GN_PARTS 16-byte records")
    sp = (ctypes.c_int64 * P)(*spatial)
    _check(_lib.tb_patch_gn_apply(_ptr_array(ptrs), _ptr_array(optrs), P, dt, N, C, sp, G, partials.data_ptr(),
                                  gamma.data_ptr() if gamma is not None else None,
                                  beta.data_ptr() if beta is not None else None, float(eps), 1 if silu else 0,
                                  _stream_handle(stream)), "tb_patch_gn_apply")
    return outs


def tb_patch_gn_apply_gathered(patches: Sequence[torch.Tensor], outs: Sequence[torch.Tensor], G: int,
                               partials: torch.Tensor, R: int, gamma: Optional[torch.Tensor],
                               beta: Optional[torch.Tensor], eps: float, silu: bool = True,
                               stream=None) -> Sequence[torch.Tensor]:
    """Normalise the local ``patches`` with the pooled statistics of ``R``
    record sets (``partials``: [R, N, G, TB_GN_PARTS, 2] int64, e.g. every
    rank's records after an all-gather)."""
    N, C, dt, spatial, ptrs = _gn_args(patches)
    P = len(patches)
    if len(outs) != P:
        raise ValueError("one output per patch")
    optrs = []
    for q, (o, t) in enumerate(zip(outs, patches)):
        _cuda_contig(o, "out %d" % q)
        if o.shape != t.shape or o.dtype != t.dtype:
            raise ValueError("out %d must match patch %d" % (q, q))
        optrs.append(o.data_ptr())
    for name, v in (("gamma", gamma), ("beta", beta)):
        if v is not None:
            _cuda_contig(v, name)
            if v.numel() != C or v.dtype != patches[0].dtype:
                raise ValueError("%s must be [C] of the patches' dtype" % name)
    _cuda_contig(partials, "partials")
    if partials.numel() * partials.element_size() != R * N * G * TB_GN_PARTS * 16:
        raise ValueError("partials must hold R*N*G*TB_GN_PARTS 16-byte records")
    sp = (ctypes.c_int64 * P)(*spatial)
    _check(_lib.tb_patch_gn_apply_gathered(_ptr_array(ptrs), _ptr_array(optrs), P, dt, N, C, sp, G,
                                           partials.data_ptr(), R, gamma.data_ptr() if gamma is not None else None,
                                           beta.data_ptr() if beta is not None else None, float(eps),
                                           1 if silu else 0, _stream_handle(stream)), "tb_patch_gn_apply_gathered")
    return outs


def patch_group_norm(patches: Sequence[torch.Tensor], G: int, gamma, beta, eps: float, silu: bool = True,
                     outs: Optional[Sequence[torch.Tensor]] = None, partials: Optional[torch.Tensor] = None,
                     stream=None) -> Sequence[torch.Tensor]:
    """Both steps: statistics of every patch, then the pooled normalisation."""
    N = patches[0].shape[0]
    if partials is None:
        partials = new_partials(len(patches), N, G, patches[0].device)
    if outs is None:
        outs = [torch.empty_like(p) for p in patches]
    tb_patch_gn_stats(patches, G, partials, stream)
    return tb_patch_gn_apply(patches, outs, G, partials, gamma, beta, eps, silu, stream)


def tb_patch_group_norm_noalloc(patches: Sequence[torch.Tensor], outs: Sequence[torch.Tensor], G: int,
                                gamma: Optional[torch.Tensor], beta: Optional[torch.Tensor], eps: float,
                                silu: bool = True, stream=None) -> Sequence[torch.Tensor]:
    """PatchGroupNorm for callers that cannot allocate device memory: the
    partial statistics live in the library's own fixed scratch array (room
    for P * N * G * TB_GN_PARTS <= TB_NOALLOC_MAX_PARTIALS records), so the
    call needs no buffer besides the inputs and outputs.  Calls share that array: order
    them on one stream.  The first call on a device looks the array's
    address up."""
    N, C, dt, spatial, ptrs = _gn_args(patches)
    P = len(patches)
    if len(outs) != P:
        raise ValueError("one output per patch")
    optrs = []
    for q, (o, t) in enumerate(zip(outs, patches)):
        _cuda_contig(o, "out %d" % q)
        if o.shape != t.shape or o.dtype != t.dtype:
            raise ValueError("out %d must match patch %d" % (q, q))
        optrs.append(o.data_ptr())
    for name, v in (("gamma", gamma), ("beta", beta)):
        if v is not None:
            _cuda_contig(v, name)
            if v.numel() != C or v.dtype != patches[0].dtype:
                raise ValueError("%s must be [C] of the patches' dtype" % name)
    sp = (ctypes.c_int64 * P)(*spatial)
    _check(_lib.tb_patch_group_norm_noalloc(_ptr_array(ptrs), _ptr_array(optrs), P, dt, N, C, sp, G,
                                            gamma.data_ptr() if gamma is not None else None,
                                            beta.data_ptr() if beta is not None else None, float(eps),
                                            1 if silu else 0, _stream_handle(stream)),
           "tb_patch_group_norm_noalloc")
    return outs


# ---------------------------------------------------------------------------
# Patchify split / patch gather
# ---------------------------------------------------------------------------

def tb_patchify_layout(extent: int, factor: int, P: int) -> Tuple[List[int], List[int]]:
    """(starts, sizes) of the P ranks' bands of an axis of ``extent``
    positions: whole bands of ``factor``, the first ranks one band more."""
    starts, sizes = (ctypes.c_int64 * max(1, P))(), (ctypes.c_int64 * max(1, P))()
    _check(_lib.tb_patchify_layout(extent, factor, P, starts, sizes), "tb_patchify_layout")
    return list(starts[:P]), list(sizes[:P])


def _shape_arr(shape) -> ctypes.Array:
    return (ctypes.c_int64 * max(1, len(shape)))(*shape)


def tb_patchify(x: torch.Tensor, axis: int, factor: int, P: int, patches: Optional[Sequence[torch.Tensor]] = None,
                slot: int = 0, stream=None) -> List[torch.Tensor]:
    """The P ranks' patches of ``x`` along ``axis``.  With ``slot`` > 0 every
    patch buffer has ``slot`` positions along the axis (the band fills the
    first ones; the rest are not written)."""
    _cuda_contig(x, "x")
    axis = axis % x.dim()
    _, sizes = tb_patchify_layout(x.shape[axis], factor, P)
    shapes = []
    for sz in sizes:
        sh = list(x.shape)
        sh[axis] = slot if slot > 0 else sz
        shapes.append(tuple(sh))
    if patches is None:
        patches = [torch.empty(sh, dtype=x.dtype, device=x.device) for sh in shapes]
    if len(patches) != P:
        raise ValueError("one patch buffer per rank")
    for q, (t, sh) in enumerate(zip(patches, shapes)):
        _cuda_contig(t, "patch %d" % q)
        if tuple(t.shape) != sh or t.dtype != x.dtype:
            raise ValueError("patch %d must be %s %s" % (q, x.dtype, sh))
    _check(_lib.tb_patchify(x.data_ptr(), _dtype_code(x), x.dim(), _shape_arr(x.shape), axis, factor, P, slot,
                            _ptr_array([t.data_ptr() for t in patches]), _stream_handle(stream)), "tb_patchify")
    return list(patches)


def tb_gather_patches(patches: Sequence[torch.Tensor], sizes: Sequence[int], axis: int,
                      out: Optional[torch.Tensor] = None, slot: int = 0, stream=None) -> torch.Tensor:
    """Concatenate the first ``sizes[p]`` positions along ``axis`` of every
    patch, in rank order.  With ``slot`` > 0 every patch buffer has ``slot``
    positions along the axis."""
    if len(patches) == 0 or len(sizes) != len(patches):
        raise ValueError("one size per patch, at least one patch")
    ref = patches[0]
    axis = axis % ref.dim()
    shape = list(ref.shape)
    shape[axis] = sum(sizes)
    for q, (t, sz) in enumerate(zip(patches, sizes)):
        _cuda_contig(t, "patch %d" % q)
        want = list(ref.shape)
        want[axis] = slot if slot > 0 else sz
        if list(t.shape) != want or t.dtype != ref.dtype:
            raise ValueError("patch %d must be %s %s" % (q, ref.dtype, tuple(want)))
    if out is None:
        out = torch.empty(shape, dtype=ref.dtype, device=ref.device)
    _cuda_contig(out, "out")
    if list(out.shape) != shape or out.dtype != ref.dtype:
        raise ValueError("out must be %s %s" % (ref.dtype, tuple(shape)))
    sz = (ctypes.c_int64 * len(sizes))(*sizes)
    _check(_lib.tb_gather_patches(_ptr_array([t.data_ptr() for t in patches]), len(patches), sz, _dtype_code(out),
                                  out.dim(), _shape_arr(shape), axis, slot, out.data_ptr(), _stream_handle(stream)),
           "tb_gather_patches")
    return out
