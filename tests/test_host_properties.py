"""Property checks of the library's host-only layout calls over random
arguments (hypothesis; no GPU, nothing is launched): every returned layout
is consistent with the oracle's geometry and with itself, and every refusal
is a status code."""
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle.geometry import axis_layout  # noqa: E402


@pytest.fixture(scope="module")
def tbl():
    from patch_groupnorm_gb300 import build
    build.build()
    from patch_groupnorm_gb300 import tileblend
    return tileblend


axis_args = st.tuples(st.integers(1, 400), st.integers(1, 96), st.sampled_from([0.0, 0.125, 0.25, 1 / 3, 0.5]),
                      st.sampled_from([1, 2, 4, 8, 16]))


def _ok_axis(a):
    ext, tile, ov, scale = a
    if int(tile * (1 - ov)) < 1:
        return None
    lay = axis_layout(ext, tile, ov, scale)
    if lay.n > 64 or lay.row_limit < 1:
        return None
    return lay


@settings(max_examples=300, deadline=None)
@given(ay=axis_args, ax=axis_args, B=st.integers(0, 4), C=st.integers(0, 4), world=st.integers(1, 9))
def test_shard_layout_partitions_the_rows_and_the_bands_match(tbl, ay, ax, B, C, world):
    ly, lx = _ok_axis(ay), _ok_axis(ax)
    if ly is None or lx is None:
        return
    shares = [tbl.tb_stitch_shard_layout(None, tbl.Axis(*ay), tbl.Axis(*ax), B, C, world, r) for r in range(world)]
    # tile rows and output rows are partitioned in rank order
    assert shares[0].row_begin == 0 and shares[-1].row_end == ly.n
    assert all(a.row_end == b.row_begin for a, b in zip(shares, shares[1:]))
    assert sum(s.out_rows for s in shares) == ly.out_extent
    assert all(s.out_row_begin == sum(t.out_rows for t in shares[:r]) for r, s in enumerate(shares))
    sizes = [s.row_end - s.row_begin for s in shares]
    assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)
    # what a rank sends is what the next rank with rows receives
    for a, b in zip(shares, shares[1:]):
        if b.row_end > b.row_begin:
            assert a.send_elems == b.halo_elems
            assert b.halo_rows == (ly.blends[b.row_begin] if b.row_begin > 0 else 0)
            assert b.halo_elems == B * C * b.halo_rows * sum(lx.extents)


@settings(max_examples=300, deadline=None)
@given(ext=st.integers(1, 600), tile=st.integers(1, 200), n=st.integers(0, 70), scale=st.sampled_from([1, 8, 16]),
       zero=st.integers(-1, 8), ramp=st.integers(0, 12))
def test_ramp_spread_accepts_exactly_the_covering_layouts(tbl, ext, tile, n, scale, zero, ramp):
    import ctypes
    from oracle.ramp import evenly_spread_origins
    org = (ctypes.c_int64 * 80)()
    a = tbl.tb_ramp_axis()
    rc = tbl._lib.tb_ramp_axis_spread(ext, tile, n, scale, zero, ramp, org, ctypes.byref(a))
    valid = (n >= 1 and tile <= ext and zero >= 0 and ramp >= 1 and (n > 1 or tile == ext) and n <= 64)
    if valid and n > 1:
        lat = [o // scale for o in evenly_spread_origins(ext, tile, n, scale)]
        valid = all(b - a_ <= tile for a_, b in zip(lat, lat[1:]))
    if not valid:
        assert rc != tbl.TB_OK
        return
    assert rc == tbl.TB_OK
    assert list(org[:n]) == evenly_spread_origins(ext, tile, n, scale)
    assert (a.n_tiles, a.tile_extent, a.out_extent, a.zero, a.ramp) == (n, tile * scale, ext * scale, zero * scale,
                                                                        ramp * scale)


@settings(max_examples=200, deadline=None)
@given(at=axis_args, ay=axis_args, ax=axis_args, B=st.integers(0, 3), C=st.integers(0, 3), world=st.integers(1, 9))
def test_frame_shard_layout_partitions_the_frames_and_the_bands_match(tbl, at, ay, ax, B, C, world):
    lt, ly, lx = _ok_axis(at), _ok_axis(ay), _ok_axis(ax)
    if lt is None or ly is None or lx is None:
        return
    shares = [tbl.tb_stitch_shard_frames_layout(tbl.Axis(*at), tbl.Axis(*ay), tbl.Axis(*ax), B, C, world, r)
              for r in range(world)]
    assert shares[0].row_begin == 0 and shares[-1].row_end == lt.n
    assert sum(s.out_rows for s in shares) == lt.out_extent
    for a, b in zip(shares, shares[1:]):
        assert a.row_end == b.row_begin
        if b.row_end > b.row_begin:
            assert a.send_elems == b.halo_elems
            assert b.halo_elems == B * C * b.halo_rows * sum(ly.extents) * sum(lx.extents)
