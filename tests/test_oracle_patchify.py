"""Pins for the ragged Patchify split and the patch gather (oracle/patchify.py):
the page's two worked row counts, a brute-force search for the only band
assignment with the properties the page states, an independent dealing
procedure, partition and round-trip identities, and the padded transfer run
through a real all-gather over gloo ranks."""
import itertools
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import patchify as PF

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_the_pages_row_counts_are_split_without_invented_rows():
    # DistVAE page, Patchify commit: 15 latent rows over 2 ranks and 16 rows
    # over 3 were padded up to 16 and 18; cut in whole rows with the extra
    # rows on the first ranks they are 8 + 7 and 6 + 5 + 5.
    assert PF.band_sizes(15, 1, 2) == [8, 7]
    assert PF.band_sizes(16, 1, 3) == [6, 5, 5]
    assert sum(PF.band_sizes(15, 1, 2)) == 15 and sum(PF.band_sizes(16, 1, 3)) == 16


def _admissible(bands, ranks):
    """Every split of `bands` into `ranks` counts that sum to it, differ by at
    most one band, and give the larger count to the earlier ranks."""
    found = []
    for counts in itertools.product(range(bands + 1), repeat=ranks):
        if sum(counts) != bands or max(counts) - min(counts) > 1:
            continue
        if any(counts[r] < counts[r + 1] for r in range(ranks - 1)):
            continue
        found.append(list(counts))
    return found


@pytest.mark.parametrize("factor", [1, 2, 8])
def test_band_sizes_are_the_only_assignment_with_the_pages_properties(factor):
    for bands in range(0, 11):
        for ranks in range(1, 5):
            only = _admissible(bands, ranks)
            assert len(only) == 1
            assert PF.band_sizes(bands * factor, factor, ranks) == [c * factor for c in only[0]]


def test_band_sizes_match_dealing_the_bands_out_in_rank_order():
    # deal band after band to rank 0, 1, ..., ranks-1, 0, 1, ...; every rank
    # then holds a contiguous run in rank order of as many bands as it was dealt
    for bands in range(0, 60):
        for ranks in range(1, 9):
            dealt = [0] * ranks
            for b in range(bands):
                dealt[b % ranks] += 1
            assert PF.band_sizes(bands * 8, 8, ranks) == [d * 8 for d in dealt]


def test_a_partial_band_and_bad_counts_are_refused():
    with pytest.raises(ValueError):
        PF.band_sizes(209, 8, 3)
    with pytest.raises(ValueError):
        PF.band_sizes(16, 1, 0)
    with pytest.raises(ValueError):
        PF.band_sizes(16, 0, 2)


def test_more_ranks_than_bands_leaves_trailing_ranks_empty():
    assert PF.band_sizes(24, 8, 5) == [8, 8, 8, 0, 0]
    starts, sizes = PF.layout(24, 8, 5)
    assert starts == [0, 8, 16, 24, 24]


@pytest.mark.parametrize("shape,axis,factor,ranks", [
    ((2, 3, 15, 7), 2, 1, 2),
    ((1, 4, 16, 9), 2, 1, 3),
    ((1, 5, 6, 40), 3, 8, 3),
    ((2, 3, 4, 24, 16), 3, 8, 2),
    ((1, 2, 3, 10, 208), 4, 8, 3),
    ((1, 2, 3, 10, 208), 2, 1, 4),
])
def test_patches_partition_the_tensor_and_gather_restores_it(shape, axis, factor, ranks):
    rng = np.random.default_rng(sum(shape) + ranks)
    x = rng.standard_normal(shape).astype(np.float32)
    patches = PF.patchify(x, axis, factor, ranks)
    sizes = PF.band_sizes(shape[axis], factor, ranks)
    assert [p.shape[axis] for p in patches] == sizes
    for p in patches:
        assert p.shape[:axis] == x.shape[:axis] and p.shape[axis + 1:] == x.shape[axis + 1:]
    # element (.., h, ..) of the tensor lies in exactly one patch, at h - start
    for start, size, p in zip(PF.band_starts(sizes), sizes, patches):
        for h in range(size):
            assert np.array_equal(np.take(p, h, axis=axis), np.take(x, start + h, axis=axis))
    assert np.array_equal(PF.gather_patches(patches, axis), x)
    # patches are copies
    if patches[0].size:
        patches[0].reshape(-1)[0] += 1.0
        assert not np.array_equal(PF.gather_patches(patches, axis), x)


def test_padding_for_the_transfer_is_sliced_off_on_the_far_side():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((2, 3, 4, 5, 208)).astype(np.float32)
    patches = PF.patchify(x, 4, 8, 3)
    sizes = [p.shape[4] for p in patches]
    slot = max(sizes)
    slots = []
    for p in patches:
        s = PF.pad_for_transfer(p, 4, slot)
        assert s.shape[4] == slot and np.array_equal(s[..., :p.shape[4]], p)
        assert not s[..., p.shape[4]:].any()
        s[..., p.shape[4]:] = 1e30            # whatever the pad holds is never read
        slots.append(s)
    assert np.array_equal(PF.gather_padded(slots, sizes, 4), x)
    with pytest.raises(ValueError):
        PF.pad_for_transfer(patches[0], 4, slot - 1)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, shape, axis, factor, q):
    # The gather as the page's ranks do it, with torch.distributed: sizes
    # first, then the payload padded to the longest patch, sliced on arrival.
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = torch.from_numpy(np.random.default_rng(11).standard_normal(shape).astype(np.float32))
        mine = torch.from_numpy(PF.patchify(x.numpy(), axis, factor, world)[rank])
        size = torch.tensor([mine.shape[axis]], dtype=torch.int64)
        sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(sizes, size)
        sizes = [int(s) for s in sizes]
        slot = max(sizes)
        pad = [0, 0] * (mine.dim() - 1 - axis) + [0, slot - mine.shape[axis]]
        sent = torch.nn.functional.pad(mine, pad)
        got = [torch.empty_like(sent) for _ in range(world)]
        dist.all_gather(got, sent)
        whole = torch.cat([g.narrow(axis, 0, s) for g, s in zip(got, sizes)], dim=axis)
        ok = torch.equal(whole, x) and sizes == PF.band_sizes(shape[axis], factor, world)
        ok = ok and np.array_equal(PF.gather_padded([g.numpy() for g in got], sizes, axis), x.numpy())
        q.put((rank, bool(ok)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,shape,axis,factor", [(2, (1, 3, 15, 6), 2, 1), (3, (1, 2, 4, 6, 208), 4, 8)])
def test_ragged_gather_over_gloo_ranks_reassembles_the_tensor(world, shape, axis, factor):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, shape, axis, factor, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert sorted(q.get(timeout=10) for _ in range(world)) == [(r, True) for r in range(world)]
