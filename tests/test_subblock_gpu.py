"""GPU parity of the SubBlock-routed forward (the SGLang Diffusion benchmark page (MiniMax-H3 on 8x H200),
section "How SubBlock Sparse Attention Works") against the CPU
oracle, through the C ABI.

Bars:
* sub-block means: fp32, |gpu - oracle| <= 2e-6 + 2e-6 |oracle| (a 16-term
  fp32 sum against an fp64 one);
* selection: identical, except for query tiles whose k-th and (k+1)-th
  oracle scores are within 1e-3 max(1, |a|, |b|). The scores are log masses,
  so an absolute 1e-3 is a 0.1% difference in mass. There any valid top-k set
  is accepted, and the output is judged against the oracle re-run with the
  GPU's set;
* bf16 output: max |gpu - oracle| <= 2e-2, mean <= 2e-3.
"""
import numpy as np
import pytest
import torch

import block_sparse_video_gb300 as bsv
from block_sparse_video_gb300.synthetic import bf16_bits, make_inputs
from oracle import subblock_oracle as so
from oracle import vsa_oracle as vo
from tests.vsa_parity import assert_errors, to_f64

pytestmark = pytest.mark.gpu

TIE = 1e-3


def _tie_tol(scores_row, k):
    s = np.sort(np.asarray(scores_row, dtype=np.float64))[::-1]
    if k >= len(s):
        return None
    a, b = s[k - 1], s[k]
    tol = TIE * max(1.0, abs(a), abs(b))
    return tol if abs(a - b) < tol else None


def _check_selection(gpu_idx, oracle_idx, scores, k):
    overrides = {}
    for t in range(oracle_idx.shape[0]):
        g = np.asarray(gpu_idx[t])
        if np.array_equal(g, oracle_idx[t]):
            continue
        tol = _tie_tol(scores[t], k)
        assert tol is not None, f"tile {t}: selection differs and is not a near-tie"
        assert len(np.unique(g)) == k and np.all(np.diff(g) > 0) and g.min() >= 0 and g.max() < len(scores[t])
        sel = np.zeros(len(scores[t]), dtype=bool)
        sel[g] = True
        s = scores[t].astype(np.float64)
        assert s[sel].min() >= s[~sel].max() - tol, f"tile {t}: gpu selection is not a top-k set"
        overrides[t] = g
    return overrides


def _run(q, k, v, lt, la, lv, sparsity):
    b, n, h, d = q.shape
    op = bsv.SubBlock(b, h, lt, la, lv, sparsity, device=q.device)
    out = op(q, k, v)
    op.check()
    views = {name: t.cpu() for name, t in op.debug_views().items()}
    return op, out, views


def _compare_head(bits, views, out, b, h, prefix, lv, sparsity, video_tiles=None, prefix_rows=None):
    args = (bits[0][b, :, h], bits[1][b, :, h], bits[2][b, :, h])
    r = so.subblock_head(*args, prefix, lv, sparsity, video_tiles=[], prefix_rows=[])
    np.testing.assert_allclose(views["sub_q"][b, h].numpy(), r["sub_q"], rtol=2e-6, atol=2e-6)
    np.testing.assert_allclose(views["sub_k"][b, h].numpy(), r["sub_k"], rtol=2e-6, atol=2e-6)
    overrides = _check_selection(views["tile_index"][b, h].numpy(), r["index"], r["scores"], r["k"])
    r = so.subblock_head(*args, prefix, lv, sparsity, video_tiles=video_tiles, prefix_rows=prefix_rows,
                         index_override=overrides)
    rows = np.where(~np.isnan(r["out"][:, 0]))[0]
    got = out[b, rows, h]
    err = np.abs(got - r["out"][rows])
    return dict(max_abs=float(err.max()) if err.size else 0.0, sum_abs=float(err.sum()),
                count=int(err.size), ties=len(overrides))


SMALL = {
    "tiny": (1, 2, 64, 64, 1024, 0.75, 30),
    "ragged_prefix_and_tail": (2, 3, 37, 50, 1000, 0.5, 31),
    "no_prefix": (1, 2, 0, 0, 700, 0.8, 32),
    "single_video_tile": (1, 2, 10, 20, 50, 0.75, 33),
    "sparsity_zero_is_dense": (1, 2, 40, 60, 640, 0.0, 34),
    "ragged_tile_with_empty_sub_blocks": (1, 2, 64, 0, 64 * 20 + 7, 0.6, 35),
    "budget_of_one_group": (1, 1, 0, 64, 64 * 40, 0.95, 36),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_shapes_full_parity(cuda_ok, name):
    b, h, lt, la, lv, s, seed = SMALL[name]
    q, k, v, _ = make_inputs(b, h, lt, la, lv, seed, device="cuda")
    _, out, views = _run(q, k, v, lt, la, lv, s)
    bits = [bf16_bits(x.cpu()) for x in (q, k, v)]
    o = to_f64(out)
    stats = [_compare_head(bits, views, o, bb, hh, lt + la, lv, s) for bb in range(b) for hh in range(h)]
    assert_errors(stats, name)


def test_medium_full_parity(cuda_ok):
    b, h, lt, la, lv, s = 1, 14, 1024, 512, 8192, 0.75
    q, k, v, _ = make_inputs(b, h, lt, la, lv, 37, device="cuda")
    _, out, views = _run(q, k, v, lt, la, lv, s)
    bits = [bf16_bits(x.cpu()) for x in (q, k, v)]
    o = to_f64(out)
    stats = [_compare_head(bits, views, o, 0, hh, lt + la, lv, s) for hh in range(h)]
    assert_errors(stats, "medium")


def _sampled(b, h, lt, la, lv, s, seed, heads, tiles_per_head):
    q, k, v, _ = make_inputs(b, h, lt, la, lv, seed, device="cuda")
    _, out, views = _run(q, k, v, lt, la, lv, s)
    bits = [bf16_bits(x.cpu()) for x in (q, k, v)]
    o = to_f64(out)
    del out, q, k, v
    t = vo.video_tile_count(lv)
    p = lt + la
    rng = np.random.default_rng(seed)
    stats = []
    for hh in heads:
        tiles = sorted(set(rng.choice(t, size=min(t, tiles_per_head), replace=False).tolist()) | {0, t - 1})
        prows = np.sort(rng.choice(p, size=min(p, 64), replace=False)) if p else np.arange(0)
        stats.append(_compare_head(bits, views, o, 0, hh, p, lv, s, video_tiles=tiles, prefix_rows=prows))
    return assert_errors(stats, f"H{h} {lt}+{la}+{lv} s={s}")


@pytest.mark.parametrize("sparsity", [0.75, 0.8])
def test_10s_shape_sampled(cuda_ok, sparsity):
    """The 10 s FastH3 shape (56 heads, 1,024 + 1,024 + 72,576 tokens), the
    launch the benchmark times; every sub-block mean and selection of three
    heads, sampled output rows."""
    _sampled(1, 56, 1024, 1024, 72576, sparsity, 38, [0, 27, 55], 12)


def test_very_long_video_smaller_router_tiles(cuda_ok):
    """T = 2,600 tiles: the router runs with 8 query tiles per CTA."""
    _sampled(1, 2, 40, 24, 64 * 2600 - 30, 0.8, 39, [1], 8)
