"""Shared parity helpers: run the CUDA path through the C ABI and compare each
intermediate and the output with the CPU oracle on the same seeded inputs.

Bars (per the method's exactness contract and the output tolerance):
* pooled statistics: fp32 means, |gpu - oracle| <= 2e-6 + 2e-6 |oracle|;
* tile selection: identical, except for query tiles whose k-th and (k+1)-th
  oracle scores differ by < 1e-3 relative. There any valid top-k set is
  accepted (every selected score >= every unselected score - tolerance), and
  the output is judged against the oracle re-run with the GPU's set;
* coarse output: |gpu - oracle| <= 1e-5 + 1e-4 |oracle|;
* bf16 output: max |gpu - oracle| <= 2e-2 and mean |gpu - oracle| <= 2e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import block_sparse_video_gb300 as bsv
from block_sparse_video_gb300.synthetic import bf16_bits, make_inputs
from oracle import vsa_oracle as vo

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
TIE_REL = 1e-3


def run_gpu(q, k, v, gate, len_text, len_audio, len_video, keep, stream=None):
    b, n, h, d = q.shape
    op = bsv.VSA(b, h, len_text, len_audio, len_video, keep, device=q.device)
    out = op(q, k, v, gate, stream=stream)
    op.check(stream)
    views = {name: t.cpu() for name, t in op.debug_views().items()}
    return op, out, views


def near_tie(scores_row, k):
    s = np.sort(np.asarray(scores_row, dtype=np.float64))[::-1]
    if k >= len(s):
        return False, 0.0
    a, b = s[k - 1], s[k]
    tol = TIE_REL * max(abs(a), abs(b))
    return abs(a - b) < tol, tol


def check_selection(gpu_idx, oracle_idx, scores, k):
    """Returns {tile: gpu selection} for accepted near-tie tiles; raises on a mismatch."""
    overrides = {}
    for t in range(oracle_idx.shape[0]):
        g = np.asarray(gpu_idx[t])
        if np.array_equal(g, oracle_idx[t]):
            continue
        tie, tol = near_tie(scores[t], k)
        assert tie, f"tile {t}: selection differs and is not a near-tie: gpu {g[:8]}.. oracle {oracle_idx[t][:8]}.."
        assert len(np.unique(g)) == k and np.all(np.diff(g) > 0) and g.min() >= 0 and g.max() < len(scores[t])
        sel = np.zeros(len(scores[t]), dtype=bool)
        sel[g] = True
        s = scores[t].astype(np.float64)
        assert s[sel].min() >= s[~sel].max() - tol, f"tile {t}: gpu selection is not a top-k set"
        overrides[t] = g
    return overrides


def compare_head(qb, kb, vb, gb, views, out_gpu, b, h, prefix, len_video, keep,
                 video_tiles=None, prefix_rows=None):
    """qb..gb: bf16 bit arrays [B, N, H, 128] (numpy uint16). out_gpu: float64 [B, N, H, 128] or a
    callable giving rows. Returns a dict of error statistics for this head."""
    args = (qb[b, :, h], kb[b, :, h], vb[b, :, h], gb[b, :, h])
    r = vo.vsa_head(*args, prefix, len_video, keep, video_tiles=[], prefix_rows=[])
    np.testing.assert_allclose(views["pooled_q"][b, h].numpy(), r["pooled_q"], rtol=2e-6, atol=2e-6)
    np.testing.assert_allclose(views["pooled_k"][b, h].numpy(), r["pooled_k"], rtol=2e-6, atol=2e-6)
    np.testing.assert_allclose(views["pooled_v"][b, h].numpy(), r["pooled_v"], rtol=2e-6, atol=2e-6)
    overrides = check_selection(views["tile_index"][b, h].numpy(), r["index"], r["scores"], r["k"])
    np.testing.assert_allclose(views["coarse"][b, h].numpy(), r["coarse"], rtol=1e-4, atol=1e-5)
    r = vo.vsa_head(*args, prefix, len_video, keep, video_tiles=video_tiles, prefix_rows=prefix_rows,
                    index_override=overrides)
    rows = np.where(~np.isnan(r["out"][:, 0]))[0]
    got = out_gpu(b, h, rows) if callable(out_gpu) else out_gpu[b, rows, h]
    err = np.abs(got - r["out"][rows])
    return dict(max_abs=float(err.max()) if err.size else 0.0, sum_abs=float(err.sum()),
                count=int(err.size), ties=len(overrides), rows=len(rows))


def assert_errors(stats, label=""):
    count = sum(s["count"] for s in stats)
    assert count > 0
    mx = max(s["max_abs"] for s in stats)
    mean = sum(s["sum_abs"] for s in stats) / count
    assert mx <= MAX_ABS, f"{label}: max abs error {mx:.3g} > {MAX_ABS}"
    assert mean <= MEAN_ABS, f"{label}: mean abs error {mean:.3g} > {MEAN_ABS}"
    return mx, mean


def to_f64(out):
    return out.float().cpu().double().numpy()


def full_check(batch, heads, len_text, len_audio, len_video, keep, seed, device="cuda"):
    """Every head, every query tile, every prefix row (small shapes)."""
    q, k, v, g = make_inputs(batch, heads, len_text, len_audio, len_video, seed, device=device)
    _, out, views = run_gpu(q, k, v, g, len_text, len_audio, len_video, keep)
    bits = [bf16_bits(x.cpu()) for x in (q, k, v, g)]
    o = to_f64(out)
    stats = [compare_head(*bits, views, o, b, h, len_text + len_audio, len_video, keep)
             for b in range(batch) for h in range(heads)]
    return assert_errors(stats, f"B{batch} H{heads} {len_text}+{len_audio}+{len_video} f={keep}")


def check_inputs(q, k, v, g, len_text, len_audio, len_video, keep, label):
    """Full parity check on caller-built inputs (small shapes)."""
    _, out, views = run_gpu(q, k, v, g, len_text, len_audio, len_video, keep)
    bits = [bf16_bits(x.cpu()) for x in (q, k, v, g)]
    o = to_f64(out)
    b_count, _, h_count, _ = q.shape
    stats = [compare_head(*bits, views, o, b, h, len_text + len_audio, len_video, keep)
             for b in range(b_count) for h in range(h_count)]
    return assert_errors(stats, label)
