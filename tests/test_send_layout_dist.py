"""The send-buffer layout of the output all-to-all, checked with real
collectives on CPU (gloo, 2 ranks).

Ulysses head sharding (the deployment "UniServe: serving FastH3 at its
fastest" describes) works like this. Each rank computes attention for its
heads over the whole sequence. The output all-to-all then returns every
sequence shard, with all heads, to its owner. Section "Fused output
combination" has the combination kernel write each row directly into its
place in the send buffer. With contiguous sequence shards, the rank-major
send buffer is the sequence order itself. So the forward writes attention
token n to row src_row[n], which is exactly what vsa_forward_rows does with
out_row_map = src_row. This test emulates that addressing on the host and
runs the all-to-all. Every rank must receive exactly its shard's rows for all
heads.
"""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

W = 2
S = 96           # sequence rows (padded length), two shards of 48
N = 80           # attention tokens (the rest is padding)
H = 4            # heads in total, 2 per rank
D = 8            # channels per head (small: this is a layout test)


def _full_output(seed=0):
    """Every head's attention output in attention-token order, and the row map."""
    rng = np.random.default_rng(seed)
    out = rng.standard_normal((N, H, D)).astype(np.float32)
    src = rng.permutation(S)[:N]      # attention token n came from sequence row src[n]
    return out, src


def _worker(rank, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=W)
    try:
        out, src = _full_output()
        h_local = H // W
        mine = out[:, rank * h_local:(rank + 1) * h_local]            # this rank's heads
        send = np.full((S, h_local, D), np.nan, dtype=np.float32)
        send[src] = mine                                              # row n -> row src[n]
        recv = torch.empty((S, h_local, D), dtype=torch.float32)
        dist.all_to_all_single(recv, torch.from_numpy(send))          # equal splits of S / W rows
        shard = recv.view(W, S // W, h_local, D).permute(1, 0, 2, 3).reshape(S // W, H, D).numpy()
        expect = np.full((S, H, D), np.nan, dtype=np.float32)
        expect[src] = out
        expect = expect[rank * (S // W):(rank + 1) * (S // W)]
        results[rank] = bool(np.array_equal(shard, expect, equal_nan=True))
    finally:
        dist.destroy_process_group()


def test_scattered_rows_form_the_output_all_to_all_send_buffer():
    port = 29500 + os.getpid() % 2000
    manager = mp.Manager()
    results = manager.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, port, results)) for r in range(W)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(results) == {0: True, 1: True}
