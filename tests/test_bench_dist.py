"""Multi-rank host logic of bench.py on CPU: two gloo ranks, each timing its own
problem; the job's step time is the max over ranks and the work is summed."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_info()
    assert (w, r) == (world, rank)
    bench.init_dist(world, "gloo")
    ms = bench.reduce_max(10.0 + rank, world)
    flops = bench.reduce_sum(1e12 * (rank + 1), world)
    bench.barrier(world)
    results[rank] = (ms, flops)
    torch.distributed.destroy_process_group()


def test_two_rank_aggregation_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        assert results[r] == (11.0, 3e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5 and bench.reduce_sum(2.0, 1) == 2.0


def test_effective_flops_matches_hand_count():
    import bench
    from block_sparse_video_gb300.synthetic import CONFIGS
    f = bench.effective_flops(CONFIGS["10s"])
    # 4*128*56*[72576*(2048 + 227*64) + 2048*74624], worked by hand
    assert f["fine"] == 4 * 128 * 56 * (72576 * (2048 + 227 * 64) + 2048 * 74624) == 38874923401216
    assert f["coarse"] == 4 * 128 * 1134 * 1134 * 56
