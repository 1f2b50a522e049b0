#!/usr/bin/env python
"""Benchmark of the VSA forward at the 10 s FastH3 shape on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload tiny|medium|5s|10s|ragged] [--keep F]

A step is one VSA forward of one DiT attention layer (tile pool, coarse
attention + top-k, fine attention with the gated combination) over the
workload of "UniServe: serving FastH3 at its fastest", section "The FastH3
workload": batch 1, 56 heads x 128, text 1,024 + audio 1,024 + video 72,576
tokens (1,134 tiles, k = 227), bf16, seeded synthetic inputs (no checkpoint).

value = effective TFLOP/s: the FLOPs the sparse pattern requires (fine
attention over the keys each query attends to, plus the coarse branch),
divided by the device time of the step, inputs resident in HBM; L2 is flushed
between timed steps. e2e = the same metric through vsa_forward_host (pinned
host buffers, host<->device copies inside the timed region), the mean over its
steps; its output is compared bit for bit with the device forward's, and a
mismatch voids the number. --workload and --keep select the other seeded
configs (tiny, medium, 5 s, and the ragged sweep at keep 0.1, 0.2 or 0.4).

Under torchrun the ranks split the layer's heads (contiguous ranges, as the
page's 4-way head sharding does; strong scaling, no collective in the data
path): each rank reads its heads in place from the full-width projections and
writes them into the same heads of the output. The step time is the max over
ranks and value counts the whole layer's FLOPs.
--impl reference times the CPU oracle on a bounded sample of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from block_sparse_video_gb300.sharding import head_ranges  # noqa: E402
from block_sparse_video_gb300.synthetic import CONFIGS, bf16_bits, make_config_inputs, make_inputs  # noqa: E402

METRIC = "VSA fwd ms/layer & effective TFLOP/s (frac of BF16 peak), 10s FastH3 shape"
UNIT = "TFLOP/s"
CFG = CONFIGS["10s"]
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def workload_config(cfg=None, keep=None):
    cfg = CFG if cfg is None else cfg
    keep = cfg.keep[0] if keep is None else keep
    t = cfg.n_video_tiles
    k = max(1, min(t, int(np.floor(keep * t + 0.5))))
    return {
        "workload": (f"VSA forward, {cfg.name} shape: B{cfg.batch} H{cfg.heads} D128, text "
                     f"{cfg.len_text} + audio {cfg.len_audio} + video {cfg.len_video} tokens "
                     f"({t} tiles of 64, k={k}, keep {keep})"),
        "batch": cfg.batch, "heads": cfg.heads, "head_dim": 128, "len_text": cfg.len_text,
        "len_audio": cfg.len_audio, "len_video": cfg.len_video, "video_tiles": t, "kept_tiles": k,
        "seed": cfg.seed,
        "l2": (f"flushed between timed steps (512 MB write); inputs "
               f"{4 * cfg.batch * (cfg.prefix + cfg.len_video) * cfg.heads * 128 * 2 / 1e9:.2f} GB"),
        "parallelism": "heads split across GPUs (contiguous ranges; 1 GPU: all heads)",
    }


def effective_flops(cfg=None, keep=None, tile_index=None):
    """FLOPs the sparse pattern requires: 4*D per (query, attended key) pair, plus
    the coarse branch (4*D per pooled query/key tile pair). Keys counted are the
    valid ones actually attended (a ragged tile counts its valid tokens)."""
    cfg = CFG if cfg is None else cfg
    keep = cfg.keep[0] if keep is None else keep
    d, p, lv = 128, cfg.prefix, cfg.len_video
    t = cfg.n_video_tiles
    n_last = lv - 64 * (t - 1)
    n = np.full(t, 64)
    n[-1] = n_last
    k = max(1, min(t, int(np.floor(keep * t + 0.5))))
    if tile_index is None:
        assert lv % 64 == 0, "ragged workloads need the selection to count keys"
        video_pairs = lv * (p + 64 * k) * cfg.batch * cfg.heads
    else:
        sel_keys = n[tile_index].sum(axis=-1)  # [B, H, T]
        video_pairs = int(((p + sel_keys) * n[None, None, :]).sum())
    prefix_pairs = p * (p + lv) * cfg.batch * cfg.heads
    fine = 4 * d * (video_pairs + prefix_pairs)
    coarse = 4 * d * t * t * cfg.batch * cfg.heads
    return {"fine": float(fine), "coarse": float(coarse), "total": float(fine + coarse)}


def kv_stream_bytes(cfg=None, keep=None):
    """K and V bytes the fine kernel moves from L2 into shared memory: every
    item (64-query tile) loads its key tiles in 128-key blocks (an odd count is
    padded with an all-zero tile that is loaded too)."""
    cfg = CFG if cfg is None else cfg
    keep = cfg.keep[0] if keep is None else keep
    t = cfg.n_video_tiles
    tp = -(-cfg.prefix // 64)
    k = max(1, min(t, int(np.floor(keep * t + 0.5))))
    blocks = cfg.batch * cfg.heads * (t * ((tp + k + 1) // 2) + tp * ((tp + t + 1) // 2))
    return float(blocks * 2 * 128 * 128 * 2)


# kernels launched by one forward: tile pool, the pooled K and V in fragment
# form, coarse attention + top-k, the fine-attention fast kernel and its exact
# redo pass
LAUNCHES_PER_FORWARD = 5


def pool_bytes(cfg=None):
    cfg = CFG if cfg is None else cfg
    return 3 * cfg.batch * cfg.len_video * cfg.heads * 128 * 2 + 3 * cfg.batch * cfg.heads * cfg.n_video_tiles * 128 * 4


def coarse_bytes(cfg=None, keep=None):
    """Algorithmic HBM bytes of the coarse + top-k step: the pooled Q, K, V read
    once (fp32), the selected tile ids (int32) and the coarse output (fp32)
    written once."""
    cfg = CFG if cfg is None else cfg
    keep = cfg.keep[0] if keep is None else keep
    bh, t = cfg.batch * cfg.heads, cfg.n_video_tiles
    k = max(1, min(t, int(math.floor(keep * t + 0.5))))
    return 3 * bh * t * 128 * 4 + bh * t * k * 4 + bh * t * 128 * 4


# fused preprocessing workload: the projections of a 10 s request arrive in a
# capacity-padded buffer of 78,080 rows (the page's preallocated size for that
# request); RoPE covers 96 of the 128 channels of each head
PRE_ROWS_IN = 78080
ROPE_DIM = 96


def preprocess_bytes(cfg=None, rope_dim=ROPE_DIM):
    """Algorithmic HBM bytes of one preprocessing launch: the N valid projection
    rows of Q/K/V/gate read once, the four packed tensors written, the RoPE
    tables read once, and the pooled Q/K/V written (padding rows are never read)."""
    cfg = CFG if cfg is None else cfg
    rows = cfg.batch * cfg.seq * cfg.heads * 128 * 2
    return 8 * rows + cfg.seq * rope_dim * 4 + 3 * cfg.batch * cfg.heads * cfg.n_video_tiles * 128 * 4


def measure_preprocess(op, cfg, dev, stream, flush, steps, warmup, peaks, world):
    """Time vsa_preprocess alone (device events, L2 flushed before each launch)
    and the fused chain vsa_preprocess + vsa_forward_preprocessed."""
    import block_sparse_video_gb300 as bsv
    from block_sparse_video_gb300.synthetic import make_norm_weights, make_projections, make_rope_tables

    rows_in = max(PRE_ROWS_IN, cfg.seq)
    proj = make_projections(cfg.batch, rows_in, cfg.heads, cfg.seed + 100, device=dev)
    wq, wk = (w.to(dev) for w in make_norm_weights(cfg.heads, cfg.seed + 101))
    cos, sin = (t.to(dev) for t in make_rope_tables(cfg.len_text, cfg.len_audio, cfg.len_video, ROPE_DIM))
    outs = [torch.empty(op.shape, dtype=torch.bfloat16, device=dev) for _ in range(4)]
    fwd_out = torch.empty(op.shape, dtype=torch.bfloat16, device=dev)
    ins = [proj[:, :, i] for i in range(4)]
    args = bsv.vsa_preprocess_args_t(
        ins[0].data_ptr(), ins[1].data_ptr(), ins[2].data_ptr(), ins[3].data_ptr(), rows_in,
        ins[0].stride(1), None, wq.data_ptr(), wk.data_ptr(), 1e-6, ROPE_DIM, 1, cos.data_ptr(),
        sin.data_ptr(), *[x.data_ptr() for x in outs])
    for _ in range(warmup):
        bsv.vsa_preprocess(op.plan, args, op.workspace)
    op.check()
    s0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    s1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        s0[i].record(stream)
        bsv.vsa_preprocess(op.plan, args, op.workspace)
        s1[i].record(stream)
    torch.cuda.synchronize(dev)
    op.check()
    pre_ms = reduce_max(statistics.mean(a.elapsed_time(b) for a, b in zip(s0, s1)), world, dev)
    for i in range(steps):
        flush.zero_()
        s0[i].record(stream)
        bsv.vsa_preprocess(op.plan, args, op.workspace)
        bsv.vsa_forward_preprocessed(op.plan, *outs, fwd_out, op.workspace)
        s1[i].record(stream)
    torch.cuda.synchronize(dev)
    op.check()
    chain_ms = reduce_max(statistics.mean(a.elapsed_time(b) for a, b in zip(s0, s1)), world, dev)
    nbytes = preprocess_bytes(cfg)
    gbs = nbytes / (pre_ms * 1e-3) / 1e9
    del proj, outs, fwd_out
    return {"ms": pre_ms, "bytes": nbytes, "GB_s": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"],
            "bound": "hbm", "rows_in": rows_in, "rope_dim": ROPE_DIM,
            "launches_timed": steps,
            "fused_chain_ms": chain_ms,
            "fused_chain": "vsa_preprocess + vsa_forward_preprocessed (coarse + top-k, fine fast, fine exact)"}


# SubBlock-routed forwards measured beside the VSA forward (the page's profiles)
SUBBLOCK_SPARSITY = (0.75, 0.8)


def subblock_keep(t, sparsity):
    """Kept key tiles: at most floor(s T) dropped, rounded up to a multiple of 8."""
    need = t - int(np.floor(sparsity * t))
    return min(t, 8 * (-(-need // 8)))


def subblock_flops(cfg, sparsity):
    """Fine FLOPs of the SubBlock pattern (4*D per attended pair; the 10 s video is
    tile-aligned) and the router's sub-block logits (2*D per sub-block pair)."""
    d, p, lv, t = 128, cfg.prefix, cfg.len_video, cfg.n_video_tiles
    k = subblock_keep(t, sparsity)
    bh = cfg.batch * cfg.heads
    fine = 4 * d * bh * (lv * (p + 64 * k) + p * (p + lv))
    router = 2 * d * bh * (4 * t) ** 2
    return k, float(fine), float(router)


def measure_subblock(q, k, v, cfg, dev, stream, flush, steps, warmup, peaks, world, sparsity):
    """Time one SubBlock-routed forward per step (sub-block pool, router, fine fast
    and exact passes) with per-stage device events, L2 flushed before each step."""
    import block_sparse_video_gb300 as bsv
    op = bsv.SubBlock(cfg.batch, cfg.heads, cfg.len_text, cfg.len_audio, cfg.len_video, sparsity, device=dev)
    out = torch.empty_like(q)
    for _ in range(warmup):
        op(q, k, v, out=out)
    op.check()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        bsv.vsa_plan_set_stage_events(op.plan, ev[i])
        op(q, k, v, out=out)
    torch.cuda.synchronize(dev)
    bsv.vsa_plan_set_stage_events(op.plan, None)
    op.check()
    stage = [reduce_max(statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev), world, dev) for j in range(3)]
    total = reduce_max(statistics.mean(e[0].elapsed_time(e[3]) for e in ev), world, dev)
    kk, fine_fl, router_fl = subblock_flops(cfg, sparsity)
    sustained = peaks["bf16_tflops_sustained"]
    del out, op
    return {"sparsity": sparsity, "kept_tiles": kk, "ms": total, "subpool_ms": stage[0],
            "router_ms": stage[1], "fine_ms": stage[2],
            "fine_TFLOP_s": fine_fl / (stage[2] * 1e-3) / 1e12,
            "fine_frac_of_bf16_sustained": fine_fl / (stage[2] * 1e-3) / 1e12 / sustained,
            "effective_TFLOP_s": fine_fl / (total * 1e-3) / 1e12,
            "router_flops": router_fl, "router_TFLOP_s": router_fl / (stage[1] * 1e-3) / 1e12,
            "launches_per_forward": 4}


# the page's 10 s request (1,000 text + 810 audio + 72,576 video tokens) inside a
# 78,080-row capacity bucket, served by one captured graph with device-side lengths
PAGE_REQUEST = (1000, 810, 72576)
CAPACITY = (1024, 1024, 76032)   # 78,080 rows


def measure_capacity(heads, dev, stream, flush, steps, warmup, world, seed):
    """Graph replay of vsa_forward_lengths for PAGE_REQUEST in a CAPACITY plan, and
    the same request through an exact-shape plan (both timed with device events,
    L2 flushed before each step)."""
    import block_sparse_video_gb300 as bsv
    from block_sparse_video_gb300.synthetic import Config
    lt, la, lv = PAGE_REQUEST
    n = lt + la + lv
    cap = bsv.VSA(1, heads, *CAPACITY, 0.2, device=dev)
    ins = make_inputs(1, heads, lt, la, lv, seed, device=dev)
    bufs = [torch.zeros(cap.shape, dtype=torch.bfloat16, device=dev) for _ in range(4)]
    for dst, src in zip(bufs, ins):
        dst[:, :n].copy_(src)
    out = torch.empty(cap.shape, dtype=torch.bfloat16, device=dev)
    lengths = torch.tensor(list(PAGE_REQUEST), dtype=torch.int64, device=dev)
    for _ in range(warmup):
        cap.forward_lengths(lengths, *bufs, out)
    cap.check()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap.forward_lengths(lengths, *bufs, out)

    def timed(fn):
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            e0[i].record(stream)
            fn()
            e1[i].record(stream)
        torch.cuda.synchronize(dev)
        return reduce_max(statistics.mean(a.elapsed_time(b) for a, b in zip(e0, e1)), world, dev)

    replay_ms = timed(graph.replay)
    cap.check()
    exact = bsv.VSA(1, heads, lt, la, lv, 0.2, device=dev)
    eout = torch.empty(exact.shape, dtype=torch.bfloat16, device=dev)
    for _ in range(warmup):
        exact(*ins, eout)
    exact_ms = timed(lambda: exact(*ins, eout))
    exact.check()
    same = bool(torch.equal(out[:, :n].view(torch.int16), eout.view(torch.int16)))
    fl = effective_flops(Config("page 10 s request", 1, heads, lt, la, lv, (0.2,), seed))["total"]
    del graph, bufs, out, eout, ins
    return {"request": {"len_text": lt, "len_audio": la, "len_video": lv}, "capacity_rows": cap.seq,
            "graph_replay_ms": replay_ms, "exact_forward_ms": exact_ms,
            "effective_TFLOP_s": fl / (replay_ms * 1e-3) / 1e12, "bitwise_equal_to_exact": same,
            "api": "vsa_forward_lengths captured once in a CUDA graph, lengths read on the device"}


def measure_send_layout(op, q, k, v, g, cfg, dev, stream, flush, steps, warmup, world, seed):
    """The forward writing each combined row through a row map into a
    78,080-row sequence-sharded send buffer (the output all-to-all's layout),
    against the plain forward on the same inputs; both timed with device
    events, L2 flushed before each step. Rows must match bit for bit."""
    from block_sparse_video_gb300.synthetic import make_row_map
    rows = max(PRE_ROWS_IN, cfg.seq)
    row_map = make_row_map(cfg.batch, cfg.seq, rows, seed).to(dev)
    send = torch.empty((cfg.batch, rows, cfg.heads, 128), dtype=torch.bfloat16, device=dev)
    plain = torch.empty(op.shape, dtype=torch.bfloat16, device=dev)
    for _ in range(warmup):
        op.forward_rows(q, k, v, g, send, row_map)
        op(q, k, v, g, plain)
    op.check()

    def timed(fn):
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            e0[i].record(stream)
            fn()
            e1[i].record(stream)
        torch.cuda.synchronize(dev)
        return reduce_max(statistics.mean(a.elapsed_time(b) for a, b in zip(e0, e1)), world, dev)

    rows_ms = timed(lambda: op.forward_rows(q, k, v, g, send, row_map))
    plain_ms = timed(lambda: op(q, k, v, g, plain))
    op.check()
    same = all(bool(torch.equal(send[b, row_map[b].long()].view(torch.int16), plain[b].view(torch.int16)))
               for b in range(cfg.batch))
    del send, plain, row_map
    return {"send_rows": rows, "forward_rows_ms": rows_ms, "plain_forward_ms": plain_ms,
            "bitwise_equal_to_plain": same,
            "api": "vsa_forward_rows: combined rows written through a random row map into the send buffer"}


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# Throttle reasons that void a timed region: it is measured again, once.
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(clocks):
    """Whether the timing rules reject a timed region: a hardware or thermal
    slowdown was active, or the SM clock sat well below its maximum with no
    reason given (a clock lock left behind). sw_power_cap alone is kept."""
    reasons = set(clocks.get("reasons") or [])
    if reasons & set(BAD_REASONS):
        return True
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    return bool(sm and smax and not reasons and sm < 0.85 * smax)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms (read only)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def reduce_max(x: float, world: int, device=None) -> float:
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int, device=None) -> float:
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


# ----------------------------------------------------------------- CPU oracle sample

def oracle_sample(n_video_tiles=256, n_prefix_rows=256, seed=None, cfg=None, keep=None):
    """Time the CPU oracle on one head of the workload: pooling, tile scores,
    selection and coarse branch for all tiles, plus fine attention for a seeded
    sample of video query tiles and prefix rows (None: all of them). Returns
    (flops, seconds, text)."""
    from oracle import vsa_oracle as vo
    cfg = CFG if cfg is None else cfg
    keep = cfg.keep[0] if keep is None else keep
    seed = cfg.seed if seed is None else seed
    q, k, v, g = make_inputs(1, 1, cfg.len_text, cfg.len_audio, cfg.len_video, seed, device="cpu")
    bits = [bf16_bits(x)[0, :, 0] for x in (q, k, v, g)]
    t = cfg.n_video_tiles
    rng = np.random.default_rng(seed)
    nt = t if n_video_tiles is None else min(t, n_video_tiles)
    npr = cfg.prefix if n_prefix_rows is None else min(cfg.prefix, n_prefix_rows)
    tiles = np.sort(rng.choice(t, size=nt, replace=False))
    prows = np.sort(rng.choice(cfg.prefix, size=npr, replace=False)) if npr else np.zeros(0, dtype=np.int64)
    t0 = time.perf_counter()
    r = vo.vsa_head(*bits, cfg.prefix, cfg.len_video, keep, video_tiles=tiles, prefix_rows=prows)
    secs = time.perf_counter() - t0
    kk = r["k"]
    n_tok = np.full(t, 64)
    n_tok[-1] = cfg.len_video - 64 * (t - 1)
    video_pairs = sum(int(n_tok[j]) * (cfg.prefix + int(n_tok[r["index"][j]].sum())) for j in tiles)
    flops = 4 * 128 * (t * t + video_pairs + len(prows) * cfg.seq)
    text = (f"1 of {cfg.heads} heads of the {cfg.name} shape (synthetic, same recipe, own seed): pool, "
            f"tile scores, top-{kk} selection and coarse branch over all {t} tiles, fine attention "
            f"for {len(tiles)} {'sampled ' if nt < t else ''}video query tiles and {len(prows)} "
            f"{'sampled ' if npr < cfg.prefix else ''}prefix rows; rate = FLOPs of that work / its wall time")
    return float(flops), secs, text


def cpu_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        blas = [i["num_threads"] for i in info if i.get("user_api") == "blas"]
        if blas:
            return int(max(blas))
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args):
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    rates, secs_all = [], []
    text = ""
    for step in range(args.warmup + args.steps):
        flops, secs, text = oracle_sample(n_video_tiles=24, n_prefix_rows=64, seed=CFG.seed + step, keep=args.keep)
        if step >= args.warmup:
            rates.append(flops / secs / 1e12)
            secs_all.append(secs)
    value = statistics.mean(rates)
    cores = cpu_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs_all),
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(CFG, args.keep),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": text},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------- GPU arm

def run_ours(args):
    import block_sparse_video_gb300 as bsv

    world, rank, local = dist_info()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    cfg = CFG
    keep = cfg.keep[0] if args.keep is None else args.keep
    peaks, peak_src = read_peaks()
    bsv.load_library()  # fails loudly if the library is not built

    # Every rank holds the whole layer's projections (same seed) and attends for its own
    # contiguous range of heads, read in place from the full-width rows and written into
    # the same heads of the full-width output; one rank takes all heads.
    h0, hr = head_ranges(cfg.heads, world)[rank]
    rcfg = dataclasses.replace(cfg, heads=hr)
    q, k, v, g = make_inputs(cfg.batch, cfg.heads, cfg.len_text, cfg.len_audio, cfg.len_video,
                             cfg.seed, device=dev)
    op = bsv.VSA(cfg.batch, hr, cfg.len_text, cfg.len_audio, cfg.len_video, keep, device=dev)
    out = torch.empty_like(q)
    hs = slice(h0, h0 + hr)
    ins = (q[:, :, hs], k[:, :, hs], v[:, :, hs], g[:, :, hs])
    out_slice = out[:, :, hs]

    def forward():
        op.forward_ex(*ins, out=out_slice)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        forward()
    op.check()
    # a partial last tile needs the selection to count the keys attended
    sel = None if cfg.len_video % 64 == 0 else op.debug_views()["tile_index"].cpu().numpy()
    fl = effective_flops(rcfg, keep, tile_index=sel)  # this rank's heads
    del sel

    steps = args.steps

    def timed_steps():
        """The timed region: K steps, L2 flushed before each, clocks sampled throughout."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        sampler = ClockSampler(local)
        barrier(world)
        torch.cuda.synchronize(dev)
        sampler.start()
        time.sleep(0.25)
        for s in range(steps):
            flush.zero_()
            bsv.vsa_plan_set_stage_events(op.plan, ev[s])
            starts[s].record(stream)
            forward()
            ends[s].record(stream)
        torch.cuda.synchronize(dev)
        clk = sampler.stop()
        barrier(world)
        bsv.vsa_plan_set_stage_events(op.plan, None)
        op.check()
        return ([starts[s].elapsed_time(ends[s]) for s in range(steps)],
                [[ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(steps)] for i in range(3)], clk)

    step_ms, stage_ms, clocks = timed_steps()
    # a region the timing rules reject (on any rank) is measured again, once
    if reduce_max(1.0 if clocks_rejected(clocks) else 0.0, world, dev) > 0:
        first = clocks
        step_ms, stage_ms, clocks = timed_steps()
        clocks = dict(clocks, remeasured=True, first_run=first)
    local_ms = statistics.mean(step_ms)
    ms = reduce_max(local_ms, world, dev)
    total_flops = reduce_sum(fl["total"], world, dev)
    value = total_flops / (ms * 1e-3) / 1e12

    pool_ms, coarse_ms, fine_ms = (reduce_max(statistics.mean(x), world, dev) for x in stage_ms)
    # per GPU: rank 0 holds the largest head share, timed against the slowest rank's kernel
    fine_tflops = fl["fine"] / (fine_ms * 1e-3) / 1e12
    sustained = peaks["bf16_tflops_sustained"]
    burst = peaks["bf16_tflops"]
    pool_gbs = pool_bytes(rcfg) / (pool_ms * 1e-3) / 1e9
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "fine_attn_traffic.json")
    if os.path.exists(tpath):
        try:
            with open(tpath) as f:
                tr = json.load(f)
            if tr.get("kernel_source_hash") == _source_hash():
                traffic = tr.get("bytes_per_launch_10s")
        except Exception:
            traffic = None

    # ---- end to end through the host-buffer entry point
    e2e = None
    if args.e2e_steps > 0:
        # this rank's heads as they arrive on the host (contiguous, pinned), and the device
        # forward's output of the same heads to check the host path against
        dev_out = out_slice.contiguous().cpu()
        hq, hk, hv, hg = [x.contiguous().cpu().pin_memory() for x in ins]
        hout = torch.empty_like(hq).pin_memory()
        dbuf = torch.empty(bsv.vsa_plan_host_path_bytes(op.plan), dtype=torch.uint8, device=dev)
        for _ in range(2):
            bsv.vsa_forward_host(op.plan, hq, hk, hv, hg, hout, dbuf)
        barrier(world)
        times = []
        for _ in range(args.e2e_steps):
            hout.fill_(float("nan"))  # outside the timed call: every step must write the whole output
            barrier(world)
            t0 = time.perf_counter()
            bsv.vsa_forward_host(op.plan, hq, hk, hv, hg, hout, dbuf)
            times.append(time.perf_counter() - t0)
        # the last step's output, bit for bit against the device forward (outside the timed region)
        same = bool(torch.equal(hout.view(torch.int16), dev_out.view(torch.int16)))
        same = reduce_max(0.0 if same else 1.0, world, dev) == 0.0
        # host wall clock, the mean over the steps (max over ranks); the median, min and max are
        # reported beside it
        e2e_s = reduce_max(statistics.mean(times), world, dev)
        tb = hq.numel() * hq.element_size()
        e2e = {"value": total_flops / e2e_s / 1e12 if same else None, "unit": UNIT, "ms_per_step": e2e_s * 1e3,
               "statistic": f"mean of {len(times)} steps",
               "median_ms": statistics.median(times) * 1e3, "min_ms": min(times) * 1e3,
               "max_ms": max(times) * 1e3, "steps_ms": [round(t * 1e3, 2) for t in times],
               "steps_over_twice_median": sum(t > 2 * statistics.median(times) for t in times),
               "bitwise_equal_to_device_forward": same,
               "h2d_bytes_per_step": int(reduce_sum(4 * tb, world, dev)),
               "d2h_bytes_per_step": int(reduce_sum(tb, world, dev)),
               "api": "vsa_forward_host (C ABI), pinned host buffers of this rank's heads, synchronous; "
                      "head groups pipelined: copy-in, forward and copy-out overlap"}
        del dev_out, hq, hk, hv, hg, hout, dbuf

    # the lines measured beside the step belong to the single-GPU benchmark workload only
    side = cfg.name == "10s" and args.keep is None and world == 1

    # ---- SubBlock-routed forwards on the same inputs (measured on their own)
    subblock = None
    if not args.no_subblock and side:
        subblock = [measure_subblock(q, k, v, cfg, dev, stream, flush, steps, args.warmup, peaks, world, s)
                    for s in SUBBLOCK_SPARSITY]

    # ---- the capacity bucket served from one graph (measured on its own)
    capacity = None
    if not args.no_capacity and side:
        capacity = measure_capacity(cfg.heads, dev, stream, flush, steps, args.warmup, world, cfg.seed + 200)

    # ---- fused preprocessing, measured on its own (not part of the forward step above)
    pre = None
    if not args.no_preprocess and side:
        pre = measure_preprocess(op, cfg, dev, stream, flush, steps, args.warmup, peaks, world)

    # ---- the combination written into the output all-to-all's send layout (measured on its own)
    send_layout = None
    if not args.no_send_layout and side:
        send_layout = measure_send_layout(op, q, k, v, g, cfg, dev, stream, flush, steps, args.warmup, world,
                                          cfg.seed + 300)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # small workloads: the oracle on one whole head; large ones: a bounded sample of one head
        whole = cfg.seq * cfg.n_video_tiles <= 10_000 * 160
        flops, secs, text = oracle_sample(None if whole else 256, None if whole else 256, cfg=cfg, keep=keep)
        rate = flops / secs / 1e12
        cpu = {"value": rate, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
               "sample": text, "seconds": secs,
               "s_per_layer_at_this_rate": fl["total"] / (rate * 1e12)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; no checkpoint)",
            "config": workload_config(cfg, keep),
            "ms_per_layer": ms,
            "effective_flops_per_step": total_flops,
            "frac_of_bf16_peak": {"sustained": value / world / sustained, "burst": value / world / burst,
                                  "source": peak_src},
            # the fine kernel is timed per launch by its own events: the burst peak applies
            "roofline": {"bound": "tensor", "kernel": "fine_attn_kernel", "achieved": fine_tflops,
                         "peak": burst, "unit": "TFLOP/s", "frac": fine_tflops / burst,
                         "traffic": traffic if cfg.name == "10s" and args.keep is None else None,
                         "peak_kind": f"bf16 dense, burst ({peak_src})",
                         "frac_of_sustained": fine_tflops / sustained, "sustained_peak": sustained,
                         "algorithmic_flops_per_launch": fl["fine"], "ms_per_launch": fine_ms},
            "kernels": {
                "pool_kernel": {"ms": pool_ms, "bytes": pool_bytes(rcfg), "GB_s": pool_gbs,
                                "frac_of_hbm": pool_gbs / peaks["hbm_gbs"]},
                "coarse_topk_kernel": {"ms": coarse_ms, "flops": fl["coarse"],
                                       "TFLOP_s": fl["coarse"] / (coarse_ms * 1e-3) / 1e12,
                                       "bytes": coarse_bytes(rcfg, keep),
                                       "frac_of_hbm": coarse_bytes(rcfg, keep) / (coarse_ms * 1e-3) / 1e9
                                       / peaks["hbm_gbs"]},
                "pool_plus_coarse": {"ms": pool_ms + coarse_ms,
                                     "bytes": pool_bytes(rcfg) + coarse_bytes(rcfg, keep),
                                     "frac_of_hbm": (pool_bytes(rcfg) + coarse_bytes(rcfg, keep))
                                     / ((pool_ms + coarse_ms) * 1e-3) / 1e9 / peaks["hbm_gbs"]},
                "fine_attn_kernel": {"ms": fine_ms, "flops": fl["fine"], "TFLOP_s": fine_tflops,
                                     "kv_l2_to_smem_bytes": kv_stream_bytes(rcfg, keep),
                                     "kv_l2_to_smem_TB_s": kv_stream_bytes(rcfg, keep) / (fine_ms * 1e-3) / 1e12},
                "preprocess_kernel": pre,
            },
            "subblock": subblock,
            "capacity_graph": capacity,
            "send_layout": send_layout,
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": LAUNCHES_PER_FORWARD * steps,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def _source_hash():
    import hashlib
    h = hashlib.sha256()
    for name in ("fine_attn.cu", "ptx.cuh", "kernels.cuh"):
        with open(os.path.join(ROOT, "block_sparse_video_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-send-layout", action="store_true",
                    help="skip the send-layout forward (vsa_forward_rows) measured beside the step")
    ap.add_argument("--no-capacity", action="store_true",
                    help="skip the separate capacity-bucket graph-replay measurement")
    ap.add_argument("--no-subblock", action="store_true",
                    help="skip the separate SubBlock-routed forward measurements")
    ap.add_argument("--no-preprocess", action="store_true",
                    help="skip the separate fused-preprocessing measurement")
    ap.add_argument("--workload", choices=list(CONFIGS), default="10s",
                    help="10s is the benchmark; the others are the seeded configs measured beside it")
    ap.add_argument("--keep", type=float, default=None,
                    help="keep fraction (default: the workload's first; the ragged sweep uses 0.1, 0.2, 0.4)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    world, _, _ = dist_info()
    if world != args.gpus and not (world == 1 and args.gpus == 1):
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
    global CFG
    CFG = CONFIGS[args.workload]
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
