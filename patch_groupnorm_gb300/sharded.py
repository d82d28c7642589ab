"""Multi-rank paths: the row-sharded stitch and the sharded PatchGroupNorm.

One process per GPU (``torch.distributed``; NCCL on GPUs).  This module holds
only the host side of the exchange steps -- who sends what to whom, and the
buffers for it; every data step runs in libtileblend's kernels through the
binding, and the messages are plain collectives or point-to-point transfers
into this GPU's own memory.

Page "Add tiled VAE parallelism & extended model support" (xDiT DistVAE
PR #14):

* halo-exchange commits: ranks exchange neighbouring rows point to point.
  For the stitch that is one message per rank boundary: rank r - 1 packs
  the raw rows its last tile row lends to rank r's first band
  (``tb_stitch_halo_pack``) and sends them; rank r stitches its rows with the
  band as a halo row (``tb_stitch2d_shard`` / ``tb_stitch3d_shard``).  The
  ranks' outputs, concatenated along the height, are the unsharded stitch,
  bit for bit.
* PatchGroupNorm fix and collective-fusion commits: the group statistics
  must be pooled over every rank's patch (mean, and the biased variance about
  the pooled mean).  The page needs two all-reduces per norm; here each rank
  writes self-describing (count, mean, M2) records of its patch
  (``tb_patch_gn_stats``), one all-gather hands every rank all records, and
  each rank normalises its own patch with the pooled statistics
  (``tb_patch_gn_apply_gathered``).

``exchange_halo`` and ``gather_partials`` carry no arithmetic and work on any
backend.  The entry points take the library binding as ``lib`` (the
default, ``tileblend``, is the only one the product uses); tests on CPU
ranks pass an object with the same calls backed by the CPU oracle, to run
this module's rank logic over gloo.
"""
from typing import List, Optional, Sequence

import torch
import torch.distributed as dist

from . import tileblend as tb


def _world_rank(group) -> (int, int):
    return dist.get_world_size(group), dist.get_rank(group)


def _global(group, r: int) -> int:
    return r if group is None else dist.get_global_rank(group, r)


def exchange_halo(send: Optional[torch.Tensor], recv: Optional[torch.Tensor], group=None) -> None:
    """Send ``send`` to the next rank and receive ``recv`` from the previous
    one (either may be None).  Non-blocking point-to-point transfers posted
    together and then waited on, so no rank waits for its successor before
    receiving from its predecessor; a rank with nothing to exchange makes no
    call (a batched exchange would need every rank of the group in it).  With
    NCCL each rank's current CUDA device must be its own GPU."""
    world, rank = _world_rank(group)
    reqs = []
    if recv is not None:
        if rank == 0:
            raise ValueError("rank 0 has no predecessor to receive from")
        reqs.append(dist.irecv(recv, _global(group, rank - 1), group=group))
    if send is not None:
        if rank + 1 >= world:
            raise ValueError("the last rank has no successor to send to")
        reqs.append(dist.isend(send, _global(group, rank + 1), group=group))
    for req in reqs:
        req.wait()


def stitch2d_row_sharded(tiles: Sequence[Sequence[torch.Tensor]], ay: tb.Axis, ax: tb.Axis, out: torch.Tensor,
                         group=None, lib=tb) -> torch.Tensor:
    """This rank's rows of a row-sharded 2D stitch.

    ``tiles[i][j]`` are the tiles of the rank's tile rows (see
    ``tb.tb_stitch_shard_layout``); ``out`` is [B, C, out_rows, W], the
    rank's slice of the full image."""
    world, rank = _world_rank(group)
    B, C = out.shape[:2]
    lay = lib.tb_stitch_shard_layout(None, ay, ax, B, C, world, rank)
    if len(tiles) != lay.row_end - lay.row_begin:
        raise ValueError("rank %d holds tile rows [%d, %d)" % (rank, lay.row_begin, lay.row_end))
    send = recv = None
    if lay.send_elems:
        send = torch.empty(lay.send_elems, dtype=out.dtype, device=out.device)
        lib.tb_stitch_halo_pack(tiles[-1], None, ay, ax, lay.row_end - 1, send)
    if lay.halo_elems:
        recv = torch.empty(lay.halo_elems, dtype=out.dtype, device=out.device)
    exchange_halo(send, recv, group)
    return lib.tb_stitch2d_shard(tiles, recv, ay, ax, lay.row_begin, lay.row_end, out)


def stitch3d_row_sharded(tiles, at: tb.Axis, ay: tb.Axis, ax: tb.Axis, out: torch.Tensor,
                         group=None, lib=tb) -> torch.Tensor:
    """This rank's rows of a video stitch sharded along the height:
    ``tiles[k][i][j]`` over all frame tiles k and the rank's tile rows i;
    ``out`` is [B, C, T, out_rows, W]."""
    world, rank = _world_rank(group)
    B, C = out.shape[:2]
    lay = lib.tb_stitch_shard_layout(at, ay, ax, B, C, world, rank)
    if any(len(per_k) != lay.row_end - lay.row_begin for per_k in tiles):
        raise ValueError("rank %d holds tile rows [%d, %d)" % (rank, lay.row_begin, lay.row_end))
    send = recv = None
    if lay.send_elems:
        send = torch.empty(lay.send_elems, dtype=out.dtype, device=out.device)
        lib.tb_stitch_halo_pack([per_k[-1] for per_k in tiles], at, ay, ax, lay.row_end - 1, send)
    if lay.halo_elems:
        recv = torch.empty(lay.halo_elems, dtype=out.dtype, device=out.device)
    exchange_halo(send, recv, group)
    return lib.tb_stitch3d_shard(tiles, recv, at, ay, ax, lay.row_begin, lay.row_end, out)


def stitch3d_frame_sharded(tiles, at: tb.Axis, ay: tb.Axis, ax: tb.Axis, out: torch.Tensor, group=None,
                           lib=tb) -> torch.Tensor:
    """This rank's frames of a video stitch sharded along the time axis:
    ``tiles[k][i][j]`` over the rank's frame tiles k and all tile rows and
    columns; ``out`` is [B, C, out_frames, H, W]."""
    world, rank = _world_rank(group)
    B, C = out.shape[:2]
    lay = lib.tb_stitch_shard_frames_layout(at, ay, ax, B, C, world, rank)
    if len(tiles) != lay.row_end - lay.row_begin:
        raise ValueError("rank %d holds frame tiles [%d, %d)" % (rank, lay.row_begin, lay.row_end))
    send = recv = None
    if lay.send_elems:
        send = torch.empty(lay.send_elems, dtype=out.dtype, device=out.device)
        lib.tb_stitch_halo_pack_frames(tiles[-1], at, ay, ax, lay.row_end - 1, send)
    if lay.halo_elems:
        recv = torch.empty(lay.halo_elems, dtype=out.dtype, device=out.device)
    exchange_halo(send, recv, group)
    return lib.tb_stitch3d_shard_frames(tiles, recv, at, ay, ax, lay.row_begin, lay.row_end, out)


def gather_partials(local: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's GroupNorm records, rank after rank: one all-gather of the
    [P, N, G, TB_GN_PARTS, 2] record buffers (all ranks hold P patches)."""
    world, _ = _world_rank(group)
    out = torch.empty((world * local.shape[0], *local.shape[1:]), dtype=local.dtype, device=local.device)
    dist.all_gather_into_tensor(out, local.contiguous(), group=group)
    return out


def patch_group_norm_sharded(patches: Sequence[torch.Tensor], G: int, gamma, beta, eps: float, silu: bool = True,
                             outs: Optional[Sequence[torch.Tensor]] = None, group=None,
                             lib=tb) -> List[torch.Tensor]:
    """GroupNorm (+ SiLU) of a tensor whose patches are spread over the ranks:
    this rank's ``patches`` come back normalised with the statistics of the
    whole tensor."""
    N = patches[0].shape[0]
    if outs is None:
        outs = [torch.empty_like(p) for p in patches]
    local = lib.new_partials(len(patches), N, G, patches[0].device)
    lib.tb_patch_gn_stats(patches, G, local)
    every = gather_partials(local, group)
    lib.tb_patch_gn_apply_gathered(patches, outs, G, every, every.shape[0], gamma, beta, eps, silu)
    return list(outs)
