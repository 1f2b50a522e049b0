"""The head split of one layer across ranks, on CPU (gloo, 2 ranks).

"UniServe: serving FastH3 at its fastest", section "The FastH3 workload":
each GPU of a 4-way sequence-parallel group attends for 14 of the 56 heads.
The forward shards by head with no exchange inside the path. These tests check
the host-side partition (every head covered exactly once, contiguous,
balanced) and that the per-rank oracle outputs, gathered over two gloo ranks,
equal the single-process oracle over all heads bit for bit.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from block_sparse_video_gb300.sharding import head_ranges

SHAPE = (1, 5, 20, 10, 200)   # batch, heads, text, audio, video (ragged last tile)
KEEP = 0.3


@pytest.mark.parametrize("heads", [1, 2, 5, 14, 56, 57, 128])
def test_head_ranges_cover_every_head_once(heads):
    for world in range(1, min(heads, 16) + 1):
        r = head_ranges(heads, world)
        assert len(r) == world
        covered = [h for h0, n in r for h in range(h0, h0 + n)]
        assert covered == list(range(heads))          # once each, in order, contiguous
        sizes = [n for _, n in r]
        assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1


def test_head_ranges_of_the_page_deployment():
    assert head_ranges(56, 4) == [(0, 14), (14, 14), (28, 14), (42, 14)]
    assert head_ranges(56, 8) == [(7 * r, 7) for r in range(8)]


@pytest.mark.parametrize("bad", [(4, 5), (0, 1), (3, 0)])
def test_head_ranges_reject_impossible_splits(bad):
    with pytest.raises(ValueError):
        head_ranges(*bad)


def _inputs():
    from block_sparse_video_gb300.synthetic import bf16_bits, make_inputs
    b, h, lt, la, lv = SHAPE
    return [bf16_bits(x) for x in make_inputs(b, h, lt, la, lv, 11, device="cpu")]


def _oracle_heads(bits, heads):
    from oracle import vsa_oracle as vo
    b, _, lt, la, lv = SHAPE
    res = vo.vsa_forward(*bits, lt, la, lv, KEEP, heads=heads)
    # [B, N, len(heads), 128] float64, heads in order
    return np.stack([np.stack([res[(bb, h)]["out"] for h in heads], axis=1) for bb in range(b)])


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    h0, n = head_ranges(SHAPE[1], world)[rank]
    mine = _oracle_heads(_inputs(), list(range(h0, h0 + n)))
    gathered = [None] * world
    torch.distributed.all_gather_object(gathered, (h0, mine))
    if rank == 0:
        results["parts"] = gathered
    torch.distributed.destroy_process_group()


def test_union_of_rank_outputs_equals_the_single_process_oracle():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    parts = sorted(results["parts"], key=lambda x: x[0])
    assert [h0 for h0, _ in parts] == [h0 for h0, _ in head_ranges(SHAPE[1], world)]
    union = np.concatenate([x for _, x in parts], axis=2)
    full = _oracle_heads(_inputs(), list(range(SHAPE[1])))
    assert union.shape == full.shape
    assert np.array_equal(union.view(np.uint64), full.view(np.uint64))   # bit for bit
