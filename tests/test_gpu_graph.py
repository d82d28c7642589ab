"""CUDA-graph replay of the sharded-decode steps (Patchify split, PatchGroupNorm
statistics and normalisation, patch gather), of the ramp stitch, of the
row-sharded stitch (halo pack and the ranks' stitches), of the video stitch
with its frame-sharded form, and of per-rank statistics with the gathered
apply, captured once and replayed with new contents at the same addresses.  Every call passes
its parameters by value, so each replay must reproduce the oracle's result
for the inputs present at replay time."""
import numpy as np
import pytest
import torch

from oracle import groupnorm as GN
from oracle import rounding as R
from oracle.ramp import ramp_stitch_2d
from patch_groupnorm_gb300 import synth
from tests.tolerance import violation

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tbl():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from patch_groupnorm_gb300 import build
    build.build()
    from patch_groupnorm_gb300 import tileblend
    return tileblend


def _within_one_ulp(got: torch.Tensor, exact: np.ndarray, dtype: str) -> bool:
    return violation(got.double().cpu().numpy(), exact, dtype) <= 1.0


def test_sharded_groupnorm_pipeline_replays_with_new_inputs(tbl):
    shape, axis, factor, ranks, G = (1, 64, 15, 24), 2, 1, 2, 8
    x = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    x.copy_(synth.normal_tensor(1, shape, "bf16"))
    gamma = synth.normal_tensor(2, (64,), "bf16").cuda() * 0.1 + 1.0
    beta = synth.normal_tensor(3, (64,), "bf16").cuda() * 0.1
    _, sizes = tbl.tb_patchify_layout(shape[axis], factor, ranks)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):   # allocate and warm up outside the capture
        parts = tbl.tb_patchify(x, axis, factor, ranks)
        outs = [torch.empty_like(p) for p in parts]
        partials = tbl.new_partials(ranks, 1, G)
        whole = torch.empty_like(x)
        tbl.tb_patch_gn_stats(parts, G, partials)
        tbl.tb_patch_gn_apply(parts, outs, G, partials, gamma, beta, 1e-6, True)
        tbl.tb_gather_patches(outs, sizes, axis, out=whole)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tbl.tb_patchify(x, axis, factor, ranks, patches=parts)
        tbl.tb_patch_gn_stats(parts, G, partials)
        tbl.tb_patch_gn_apply(parts, outs, G, partials, gamma, beta, 1e-6, True)
        tbl.tb_gather_patches(outs, sizes, axis, out=whole)
    for seed in (21, 22, 23):
        fresh = synth.normal_tensor(seed, shape, "bf16") * (1.0 + seed % 3) + (seed - 22)
        x.copy_(fresh.to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        exact = GN.patch_group_norm([x.double().cpu().numpy()], G, gamma.double().cpu().numpy(),
                                    beta.double().cpu().numpy(), 1e-6, silu=True)[0]
        assert _within_one_ulp(whole, exact, "bf16"), seed


def test_ramp_stitch_replays_with_new_inputs(tbl):
    ay = tbl.RampAxis.spread(64, 32, 3, 8)
    ax = tbl.RampAxis.spread(96, 32, 5, 8)
    shape = (1, 2, ay.tile_extent, ax.tile_extent)
    tiles = [[torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in ax.origins] for _ in ay.origins]
    out = torch.empty((1, 2, ay.out_extent, ax.out_extent), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tbl.tb_stitch2d_ramp(tiles, ay, ax, out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tbl.tb_stitch2d_ramp(tiles, ay, ax, out)
    rng = np.random.default_rng(5)
    for _ in range(3):
        host = [[torch.from_numpy(rng.uniform(-1, 1, shape)).to(torch.bfloat16) for _ in ax.origins]
                for _ in ay.origins]
        for rd, rh in zip(tiles, host):
            for td, th in zip(rd, rh):
                td.copy_(th)
        g.replay()
        torch.cuda.synchronize()
        exact = ramp_stitch_2d([[t.double().numpy() for t in row] for row in host], ay.origins, ax.origins,
                               ay.tile_extent, ax.tile_extent, (ay.out_extent, ax.out_extent), ay.zero, ay.ramp,
                               ax.zero, ax.ramp)
        assert _within_one_ulp(out, exact, "bf16")


def test_row_sharded_stitch_replays_with_new_inputs(tbl):
    # two ranks' shares of a row-sharded stitch run one after the other on
    # this GPU: rank 0 packs the band its last tile row lends (halo pack) into
    # the buffer the exchange would deliver to rank 1, and each rank stitches
    # its own tile rows; pack and stitches captured once, replayed with new
    # tiles, must equal the unsharded stitch of those tiles bit for bit
    from oracle.geometry import axis_layout
    ay, ax = tbl.Axis(48, 16, 0.25, 8), tbl.Axis(40, 16, 0.25, 8)
    ly = axis_layout(48, 16, 0.25, 8)
    lx = axis_layout(40, 16, 0.25, 8)
    B, C = 1, 3
    tiles = [[torch.empty((B, C, hy, wx), dtype=torch.bfloat16, device="cuda") for wx in lx.extents]
             for hy in ly.extents]
    lays = [tbl.tb_stitch_shard_layout(None, ay, ax, B, C, 2, r) for r in range(2)]
    assert lays[0].send_elems > 0 and lays[1].halo_elems == lays[0].send_elems
    band = torch.empty(lays[0].send_elems, dtype=torch.bfloat16, device="cuda")
    outs = [torch.empty((B, C, lay.out_rows, lx.out_extent), dtype=torch.bfloat16, device="cuda") for lay in lays]
    whole = torch.empty((B, C, ly.out_extent, lx.out_extent), dtype=torch.bfloat16, device="cuda")

    def ranks():
        l0, l1 = lays
        tbl.tb_stitch_halo_pack(tiles[l0.row_end - 1], None, ay, ax, l0.row_end - 1, band)
        tbl.tb_stitch2d_shard(tiles[l0.row_begin:l0.row_end], None, ay, ax, l0.row_begin, l0.row_end, outs[0])
        tbl.tb_stitch2d_shard(tiles[l1.row_begin:l1.row_end], band, ay, ax, l1.row_begin, l1.row_end, outs[1])

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ranks()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ranks()
    rng = np.random.default_rng(9)
    for _ in range(3):
        for row in tiles:
            for t in row:
                t.copy_(torch.from_numpy(rng.uniform(-1, 1, tuple(t.shape))).to(torch.bfloat16))
        band.fill_(float("nan"))
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        tbl.tb_stitch2d(tiles, ay, ax, whole)
        torch.cuda.synchronize()
        assert torch.equal(torch.cat(outs, dim=2).view(torch.int16), whole.view(torch.int16))


def test_video_stitch_and_frame_sharded_stitch_replay_with_new_inputs(tbl):
    # tb_stitch3d, and two ranks' shares of the same video sharded along the
    # frames (frame-band pack + each rank's stitch), in one graph; replayed
    # with new tiles: the stitch equals the oracle and the ranks' outputs
    # concatenated equal the stitch, bit for bit
    from oracle.geometry import axis_layout
    from oracle.stitch import stitch as oracle_stitch
    from tests.stitch_helpers import to_storage
    geo = [(17, 8, 0.25, 1), (24, 8, 0.25, 8), (20, 8, 0.25, 8)]
    at, ay, ax = (tbl.Axis(*a) for a in geo)
    lt, ly, lx = (axis_layout(*a) for a in geo)
    B, C = 1, 2
    tiles = [[[torch.empty((B, C, ft, hy, wx), dtype=torch.bfloat16, device="cuda") for wx in lx.extents]
              for hy in ly.extents] for ft in lt.extents]
    whole = torch.empty((B, C, lt.out_extent, ly.out_extent, lx.out_extent), dtype=torch.bfloat16, device="cuda")
    lays = [tbl.tb_stitch_shard_frames_layout(at, ay, ax, B, C, 2, r) for r in range(2)]
    assert lays[0].send_elems > 0 and lays[1].halo_elems == lays[0].send_elems
    band = torch.empty(lays[0].send_elems, dtype=torch.bfloat16, device="cuda")
    outs = [torch.empty((B, C, lay.out_rows, ly.out_extent, lx.out_extent), dtype=torch.bfloat16, device="cuda")
            for lay in lays]

    def run():
        l0, l1 = lays
        tbl.tb_stitch3d(tiles, at, ay, ax, whole)
        tbl.tb_stitch_halo_pack_frames(tiles[l0.row_end - 1], at, ay, ax, l0.row_end - 1, band)
        tbl.tb_stitch3d_shard_frames(tiles[l0.row_begin:l0.row_end], None, at, ay, ax, l0.row_begin, l0.row_end,
                                     outs[0])
        tbl.tb_stitch3d_shard_frames(tiles[l1.row_begin:l1.row_end], band, at, ay, ax, l1.row_begin, l1.row_end,
                                     outs[1])

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    rng = np.random.default_rng(17)
    for _ in range(2):
        host = [[[torch.from_numpy(rng.uniform(-1, 1, tuple(t.shape))).to(torch.bfloat16) for t in row]
                 for row in frame] for frame in tiles]
        for fd, fh in zip(tiles, host):
            for rd, rh in zip(fd, fh):
                for td, th in zip(rd, rh):
                    td.copy_(th)
        for buf in [whole, band, *outs]:
            buf.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_stitch([[[to_storage(t, "bf16") for t in row] for row in frame] for frame in host],
                            [lt, ly, lx], "bf16")
        assert np.array_equal(to_storage(whole.cpu(), "bf16"), ref)
        assert torch.equal(torch.cat(outs, dim=2).view(torch.int16), whole.view(torch.int16))


def test_gathered_groupnorm_replays_with_new_inputs(tbl):
    # two ranks' statistics calls writing their record sets side by side (as
    # an all-gather lays them out) and each rank's gathered apply, in one
    # graph; replayed with new patches, within the GroupNorm tolerance
    from tests.tolerance import gn_violation
    G = 8
    shape = (1, 32, 20, 48)
    parts = [torch.empty((1, 32, h, 48), dtype=torch.bfloat16, device="cuda") for h in (8, 12)]
    gamma = (synth.normal_tensor(4, (32,), "bf16") * 0.1 + 1.0).cuda()
    beta = (synth.normal_tensor(5, (32,), "bf16") * 0.1).cuda()
    every = tbl.new_partials(2, 1, G)
    outs = [torch.empty_like(p) for p in parts]

    def run():
        for r in range(2):
            tbl.tb_patch_gn_stats([parts[r]], G, every[r:r + 1])
        for r in range(2):
            tbl.tb_patch_gn_apply_gathered([parts[r]], [outs[r]], G, every, 2, gamma, beta, 1e-6, True)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    for seed in (31, 32):
        x = synth.normal_tensor(seed, shape, "bf16") * (1.0 + seed % 2) + (seed - 31.5)
        cpu = [p.contiguous() for p in torch.split(x.to(torch.bfloat16), [8, 12], dim=2)]
        for d, c in zip(parts, cpu):
            d.copy_(c)
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        with np.errstate(over="ignore"):
            assert gn_violation([o.cpu() for o in outs], cpu, gamma.cpu(), beta.cpu(), G, 1e-6, True, "bf16") <= 1.0
