"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Small shapes are checked on every head, query tile and prefix row, including
the degenerate cases (empty prefix, non-64-aligned prefix, ragged last video
tile, a single video tile, a single video token, k = 1, k = T). The workload
sizes run in the same launch configuration the benchmark times and are
checked on every pooled statistic, selection and coarse row of a seeded
sample of heads and on a seeded sample of output rows.
"""
import gc

import numpy as np
import pytest
import torch

import block_sparse_video_gb300 as bsv
from block_sparse_video_gb300.synthetic import CONFIGS, bf16_bits, make_config_inputs, make_inputs
from oracle import vsa_oracle as vo
from tests.vsa_parity import assert_errors, check_inputs, compare_head, full_check, run_gpu, to_f64

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": (1, 2, 64, 64, 1024, 0.2, 0),
    "ragged_prefix_and_tail": (2, 3, 37, 50, 1000, 0.3, 5),
    "no_prefix": (1, 2, 0, 0, 700, 0.25, 6),
    "single_video_tile": (1, 2, 10, 20, 50, 0.2, 7),
    "keep_all_is_dense": (1, 2, 40, 60, 640, 1.0, 8),
    "k_is_one": (1, 2, 64, 0, 2048, 0.01, 9),
    "one_video_token": (1, 1, 3, 2, 1, 0.2, 10),
    "text_only_prefix": (1, 4, 130, 0, 4096, 0.2, 11),
    "odd_tile_count": (1, 3, 64, 64, 64 * 37 + 5, 0.2, 12),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_shapes_full_parity(cuda_ok, name):
    full_check(*SMALL[name])


@pytest.mark.parametrize("keep", [0.1, 0.2, 0.4])
def test_ragged_sweep_scaled_down_full_parity(cuda_ok, keep):
    """The ragged sparsity sweep's structure at a size the oracle checks in full:
    batch 2, a 1,000 + 700 token prefix (not a multiple of 64), 8,100 video
    tokens (127 tiles, the last with 36 tokens), keep 0.1 / 0.2 / 0.4 (k = 13,
    25, 51). Every head, query tile, prefix row and selection."""
    full_check(2, 2, 1000, 700, 8100, keep, 41)


def test_medium_full_parity(cuda_ok):
    c = CONFIGS["medium"]
    full_check(c.batch, c.heads, c.len_text, c.len_audio, c.len_video, c.keep[0], c.seed)


def _sampled(q, k, v, g, lt, la, lv, keep, pairs, tiles_per_head, prefix_pairs, seed):
    _, out, views = run_gpu(q, k, v, g, lt, la, lv, keep)
    bits = [bf16_bits(x.cpu()) for x in (q, k, v, g)]
    out_cpu = out.cpu()
    del out
    t = vo.video_tile_count(lv)
    p = lt + la
    rng = np.random.default_rng(seed)
    stats = []
    for (b, h) in pairs:
        tiles = set(rng.choice(t, size=min(t, tiles_per_head), replace=False).tolist()) | {0, t - 1}
        if (b, h) in prefix_pairs:
            prows = np.arange(p)
        else:
            prows = np.sort(rng.choice(p, size=min(p, 64), replace=False)) if p else np.arange(0)
        stats.append(compare_head(*bits, views, lambda bb, hh, rows: out_cpu[bb, rows, hh].double().numpy(),
                                  b, h, p, lv, keep, video_tiles=sorted(tiles), prefix_rows=prows))
    return stats


def _pairs(batch, heads, n, seed):
    rng = np.random.default_rng(seed)
    allp = [(b, h) for b in range(batch) for h in range(heads)]
    pick = rng.choice(len(allp), size=min(n, len(allp)), replace=False)
    return [allp[i] for i in sorted(pick)]


@pytest.mark.parametrize("name", ["5s", "10s"])
def test_workload_sampled_parity(cuda_ok, name):
    c = CONFIGS[name]
    q, k, v, g = make_config_inputs(c, device="cuda")
    pairs = _pairs(c.batch, c.heads, 6 if name == "10s" else 4, c.seed)
    stats = _sampled(q, k, v, g, c.len_text, c.len_audio, c.len_video, c.keep[0], pairs, 24,
                     set(pairs[:1]), c.seed)
    del q, k, v, g
    gc.collect()
    torch.cuda.empty_cache()
    assert_errors(stats, name)


def test_ragged_sweep_sampled_parity(cuda_ok):
    c = CONFIGS["ragged"]
    q, k, v, g = make_config_inputs(c, device="cuda")
    for i, keep in enumerate(c.keep):
        pairs = _pairs(c.batch, c.heads, 3, c.seed + i)
        stats = _sampled(q, k, v, g, c.len_text, c.len_audio, c.len_video, keep, pairs, 16,
                         set(pairs[:1]) if i == 0 else set(), c.seed + i)
        assert_errors(stats, f"ragged f={keep}")
    del q, k, v, g
    gc.collect()
    torch.cuda.empty_cache()


def test_long_video_smaller_coarse_tiles(cuda_ok):
    """T = 1,500 video tiles: the tcgen05 coarse kernel holds each score row in
    72 registers a lane (its widest row form)."""
    q, k, v, g = make_inputs(1, 2, 40, 24, 96000, 21, device="cuda")
    stats = _sampled(q, k, v, g, 40, 24, 96000, 0.2, [(0, 0), (0, 1)], 24, {(0, 1)}, 21)
    assert_errors(stats, "long video")


def test_very_long_video_sixteen_coarse_tiles(cuda_ok):
    """T = 2,600 video tiles (the last one ragged), past the tcgen05 coarse
    kernel's 2,304: the mma.sync coarse kernel keeps 16 query tiles per CTA
    (its score rows would not fit 32). Every pooled statistic, selection and
    coarse row of both heads is checked."""
    lv = 64 * 2600 - 30
    q, k, v, g = make_inputs(1, 2, 40, 24, lv, 23, device="cuda")
    stats = _sampled(q, k, v, g, 40, 24, lv, 0.2, [(0, 0), (0, 1)], 16, {(0, 0)}, 23)
    assert_errors(stats, "very long video")


def test_longest_video_eight_coarse_tiles(cuda_ok):
    """T = 4,000 video tiles: the mma.sync coarse kernel keeps 8 query tiles per
    CTA and runs its tensor-core tiles with half the rows empty."""
    lv = 64 * 4000 - 17
    q, k, v, g = make_inputs(1, 1, 64, 0, lv, 24, device="cuda")
    stats = _sampled(q, k, v, g, 64, 0, lv, 0.2, [(0, 0)], 12, {(0, 0)}, 24)
    assert_errors(stats, "longest video")


def test_deterministic(cuda_ok):
    c = CONFIGS["medium"]
    q, k, v, g = make_config_inputs(c, device="cuda")
    op = bsv.VSA(c.batch, c.heads, c.len_text, c.len_audio, c.len_video, c.keep[0])
    a = op(q, k, v, g).clone()
    ia = op.debug_views()["tile_index"].clone()
    b = op(q, k, v, g)
    op.check()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(ia, op.debug_views()["tile_index"])


@pytest.mark.parametrize("heads,subblock,pinned", [(2, False, True), (11, False, True), (11, True, True),
                                                    (1, False, True), (24, False, True), (24, False, False),
                                                    (11, True, False), (24, False, "inputs")])
def test_host_buffer_path_matches_device_path(cuda_ok, heads, subblock, pinned):
    """The host-buffer path copies head groups in, runs each group's forward and
    copies it out, pipelined. Group widths ramp up and end on two heads: 11
    heads run as groups of 4, 6 and 1; 24 heads as 4, 6, 8, 4 and 2; 2 heads as
    two of one. With pinned inputs the first group is gathered by a kernel
    reading host memory, and with a pinned output the last group is written by
    a kernel; pageable buffers (all of them, or the output alone) go through
    strided copies. Every head's result must equal the device path bit for
    bit."""
    lt, la, lv = 64, 37, 1000
    q, k, v, g = make_inputs(1, heads, lt, la, lv, 0, device="cuda")
    op = bsv.SubBlock(1, heads, lt, la, lv, 0.6) if subblock else bsv.VSA(1, heads, lt, la, lv, 0.2)
    dev = op(q, k, v, None if subblock else g)
    op.check()
    host = [x.cpu() for x in (q, k, v, g)]
    hout = torch.full_like(host[0], float("nan"))
    if pinned:
        host = [x.pin_memory() for x in host]
        if pinned is True:
            hout = hout.pin_memory()
    hq, hk, hv, hg = host
    buf = torch.empty(bsv.vsa_plan_host_path_bytes(op.plan), dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call reuses the pipeline's streams and events
        bsv.vsa_forward_host(op.plan, hq, hk, hv, None if subblock else hg, hout, buf)
        assert torch.equal(hout.view(torch.int16), dev.cpu().view(torch.int16))
        hout.fill_(float("nan"))


def test_exact_ties_at_the_cut_take_the_lower_tiles(cuda_ok):
    """Scores tie exactly at the cut: every video query is the all-ones vector
    and every key tile is constant, so s[t][j] = c_j * sqrt(128) for all t,
    bit-equal for equal c_j on both sides. Five tiles score highest and four
    tie for the sixth place (k = 6 of 30 tiles): no threshold separates k
    scores, the selection takes the lowest-index tied tile (the oracle's rule),
    and the output matches the oracle."""
    lt, la, lv, keep = 20, 12, 64 * 30, 0.2
    q, k, v, g = make_inputs(1, 2, lt, la, lv, 40, device="cuda")
    t_count = lv // 64
    c = [-(j + 1) / 64.0 for j in range(t_count)]     # distinct, all below the groups
    for j in (20, 21, 22, 23, 24):
        c[j] = 1.0                                       # the top five
    for j in (2, 9, 14, 27):
        c[j] = 0.5                                       # tied for the sixth place
    p = lt + la
    q[:, p:] = 1.0
    for j in range(t_count):
        k[:, p + 64 * j: p + 64 * (j + 1)] = c[j]
    assert vo.keep_count(t_count, keep) == 6
    _, _, views = run_gpu(q, k, v, g, lt, la, lv, keep)
    expect = np.array([2, 20, 21, 22, 23, 24])
    idx = views["tile_index"].numpy()
    assert (idx == expect).all(), idx[0, 0, :3]
    check_inputs(q, k, v, g, lt, la, lv, keep, "exact ties at the cut")


def test_stage_events_time_each_kernel(cuda_ok):
    q, k, v, g = make_inputs(1, 2, 64, 64, 1024, 0, device="cuda")
    op = bsv.VSA(1, 2, 64, 64, 1024, 0.2)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    bsv.vsa_plan_set_stage_events(op.plan, ev)
    op(q, k, v, g)
    op.check()
    bsv.vsa_plan_set_stage_events(op.plan, None)
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
    assert all(t > 0 for t in times)


@pytest.mark.parametrize("level", [6.0, 16.0])
def test_large_score_jump_after_first_block(cuda_ok, level):
    """One video key tile scores far above everything in the first key block
    (2^94 and 2^261 in softmax units): the fast pass's fixed reference cannot
    hold it, so the kernel must rerun those items with exact rescaling."""
    lt, la, lv = 40, 24, 1024
    q, k, v, g = make_inputs(1, 2, lt, la, lv, 31, device="cuda")
    q.fill_(1.0)
    k[:, lt + la + 5 * 64: lt + la + 6 * 64] = level
    check_inputs(q, k, v, g, lt, la, lv, 0.2, f"score jump {level}")


def test_uniformly_low_scores_use_the_exact_pass(cuda_ok):
    """Every score sits between about -130 and -146 in softmax (log2) units. Against the
    fast pass's fixed reference every P would underflow, so the floor on the row sums
    must send every item to the exact pass, which rescales to the running maximum.
    Video tile j's keys are one bf16 step (1/16) above tile j-1's, so the coarse
    scores are distinct and the selection has no near-tie."""
    lt, la, lv = 40, 24, 1024
    q, k, v, g = make_inputs(1, 2, lt, la, lv, 37, device="cuda")
    q.fill_(-1.0)
    k.mul_(0.02).add_(8.0)
    p = lt + la
    for j in range(lv // 64):
        k[:, p + 64 * j: p + 64 * (j + 1)] += 0.0625 * j
    check_inputs(q, k, v, g, lt, la, lv, 0.2, "uniformly low scores")
