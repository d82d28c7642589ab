"""Oracle geometry against hand-typed tables (tests/golden/geometry.json)."""
import json
import os

import pytest

from oracle.geometry import axis_layout

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "geometry.json")
CASES = json.load(open(GOLDEN))["cases"]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_axis_layout_matches_golden(case):
    lay = axis_layout(case["latent_extent"], case["latent_tile"], case["overlap"], case["scale"])
    assert lay.stride == case["stride"]
    assert lay.blend_extent == case["blend_extent"]
    assert lay.row_limit == case["row_limit"]
    assert lay.extents == case["extents"]
    assert lay.blends == case["blends"]
    assert lay.kept == case["kept"]
    assert lay.out_extent == case["out_extent"]
    if "origins_px" in case:
        assert [o * case["scale"] for o in lay.origins] == case["origins_px"]
    if "decoded_latents_per_side" in case:
        assert sum(lay.extents) // case["scale"] == case["decoded_latents_per_side"]
        assert lay.n == case["tiles_per_side"]


def test_offsets_are_prefix_sums_of_kept():
    lay = axis_layout(200, 120, 0.25, 8)
    assert lay.offsets == [0, 720, 1440]


def test_canvas_within_one_tile_is_one_tile():
    lay = axis_layout(40, 64, 0.25, 8)
    assert lay.n == 1 and lay.extents == [320] and lay.blends == [0] and lay.out_extent == 320


def test_zero_overlap_has_no_blend_and_keeps_whole_tiles():
    lay = axis_layout(100, 32, 0.0, 8)
    assert lay.stride == 32 and lay.blend_extent == 0 and lay.row_limit == 256
    assert lay.blends == [0, 0, 0, 0] and lay.kept == lay.extents and lay.out_extent == 800


def test_explicit_blend_and_limit_override_stock():
    lay = axis_layout(128, 64, 0.25, 8, blend_extent=64, row_limit=448)
    assert lay.blends == [0, 64, 64] and lay.kept == [448, 448, 256]
