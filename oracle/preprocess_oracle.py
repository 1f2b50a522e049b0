"""CPU oracle for the fused attention preprocessing in front of the VSA forward.

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import or run it; the library never does.
It shares no code with the CUDA path.

What it computes follows "UniServe: serving FastH3 at its fastest", section
"Fused attention preprocessing". One pass over the projected Q/K/V/gate rows
does the following:

* learned Q/K RMSNorm;
* partial RoPE;
* tile pooling over valid tokens, into FP32 pooled statistics;
* tile packing, i.e. gathering the valid rows of a capacity-padded projection
  buffer into the attention layout, so that padding never reaches a later
  step;
* copying the gate.

Section "The Kernel Layer" of the SGLang Diffusion benchmark page (MiniMax-H3 on 8x H200)
gives the RoPE width used there (96 of the 128
channels of a head). It also says that the fused norm + RoPE kernel rounds the
normalised value before applying RoPE.

Readings of what the page leaves open (each is listed with its reason in the
design notes):

* RMSNorm runs per token and head over the 128 channels of that head. Under
  head sharding, a norm over all heads would need heads held on other GPUs.
  y = x / sqrt(mean(x^2) + eps) * w, with one learned weight per (head,
  channel) for Q and another for K.
* RoPE rotates channels [0, rope_dim) of every head and passes the rest
  through. Pairs are (2i, 2i+1) ("interleaved") or (i, i + rope_dim/2) ("half
  split"). The pair (a, b) at token n becomes
  (a cos - b sin, a sin + b cos), i.e. a + ib multiplied by e^{i theta}.
  cos and sin come from caller-supplied per-token tables of rope_dim/2 angles.
  Tables can encode 3-D positions with any split of the angles over axes.
* Rounding: the normalised value is rounded to bf16, RoPE is applied to the
  rounded value, and the result is rounded to bf16 (RNE).
* Packing: attention token n of batch b reads projection row src_row[b, n]
  of that batch. An index outside the buffer gives a zero row and is
  reported. No map means row n.
* Pooled statistics are means of the packed bf16 outputs (the values attention
  reads) over each video tile's valid tokens, as in the forward.

Arithmetic is fp64 apart from the two stated roundings to bf16.
"""
from __future__ import annotations

import numpy as np

from oracle import vsa_oracle as vo

HEAD_DIM = 128


def round_bf16(x) -> np.ndarray:
    """Round to the nearest bf16 value, ties to even, directly from fp64 (bf16:
    8 significant bits, fp32's exponent range). Returns the values as fp64."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                 # |x| in [2**(e-1), 2**e)
    e = np.maximum(e, -125)            # spacing is fixed at 2**-133 below the smallest normal
    step = np.ldexp(1.0, e - 8)
    return np.rint(x / step) * step    # rint: halves to even; scaling by 2**k is exact


def rms_norm(x, w, eps: float) -> np.ndarray:
    """RMSNorm of each row over its 128 channels: x / sqrt(mean(x^2) + eps) * w."""
    x = np.asarray(x, dtype=np.float64)
    ms = (x * x).mean(axis=-1, keepdims=True)
    return x / np.sqrt(ms + float(eps)) * np.asarray(w, dtype=np.float64)


def rope_pairs(rope_dim: int, interleaved: bool):
    """Channel indices (first, second) of the rotated pairs, pair i using angle i."""
    half = rope_dim // 2
    i = np.arange(half)
    if interleaved:
        return 2 * i, 2 * i + 1
    return i, i + half


def rope(x, cos, sin, rope_dim: int, interleaved: bool) -> np.ndarray:
    """Rotary embedding on channels [0, rope_dim) of each row. Row n's pair i is
    rotated by the angle whose cosine and sine are cos[n, i], sin[n, i]. The
    remaining channels are unchanged."""
    x = np.array(x, dtype=np.float64)
    if rope_dim == 0:
        return x
    a_idx, b_idx = rope_pairs(rope_dim, interleaved)
    c = np.asarray(cos, dtype=np.float64)
    s = np.asarray(sin, dtype=np.float64)
    a = x[..., a_idx].copy()
    b = x[..., b_idx].copy()
    x[..., a_idx] = a * c - b * s
    x[..., b_idx] = a * s + b * c
    return x


def gather_rows(proj, src_row, n_rows: int):
    """Rows of one batch's projection buffer [S_in, ...] in attention order.
    Returns (rows [n_rows, ...], bad) where bad marks map entries outside
    [0, S_in); those rows are zero."""
    proj = np.asarray(proj)
    s_in = proj.shape[0]
    src = np.arange(n_rows) if src_row is None else np.asarray(src_row, dtype=np.int64)
    bad = (src < 0) | (src >= s_in)
    out = np.zeros((n_rows,) + proj.shape[1:], dtype=np.float64)
    ok = ~bad
    out[ok] = proj[src[ok]]
    return out, bad


def preprocess_rows(q, k, v, gate, wq, wk, eps, cos, sin, rope_dim, interleaved):
    """The per-token work of one head: rows [n, 128] of packed (gathered) Q, K,
    V, gate values. Returns bf16-valued fp64 arrays (q_out, k_out, v_out, g_out)."""
    qn = round_bf16(rms_norm(q, wq, eps))
    kn = round_bf16(rms_norm(k, wk, eps))
    q_out = round_bf16(rope(qn, cos, sin, rope_dim, interleaved))
    k_out = round_bf16(rope(kn, cos, sin, rope_dim, interleaved))
    return q_out, k_out, np.array(v, dtype=np.float64), np.array(gate, dtype=np.float64)


def preprocess(q_in, k_in, v_in, g_in, prefix: int, len_video: int, wq, wk, eps: float,
               cos, sin, rope_dim: int, interleaved: bool = True, src_row=None,
               heads=None):
    """Fused attention preprocessing over capacity-padded projections.

    q_in, k_in, v_in, g_in: [B, S_in, H, 128] bf16 values (bit patterns or floats).
    src_row: None or int [B, N], the projection row of each attention token.
    wq, wk: [H, 128] RMSNorm weights. cos, sin: [N, rope_dim / 2].
    heads: heads to compute (default all; the others stay NaN).

    Returns a dict of the following:
    * q, k, v, gate: [B, N, H, 128] fp64 holding bf16 values;
    * pooled_q, pooled_k, pooled_v: fp32 [B, H, T, 128];
    * bad: bool [B, N], map entries outside the buffer.
    """
    q_in, k_in, v_in, g_in = (vo.widen(x) for x in (q_in, k_in, v_in, g_in))
    b_count, _, h_count, d = q_in.shape
    assert d == HEAD_DIM and rope_dim % 2 == 0 and 0 <= rope_dim <= HEAD_DIM
    n = int(prefix) + int(len_video)
    t_count = vo.video_tile_count(len_video)
    out = {name: np.full((b_count, n, h_count, d), np.nan) for name in ("q", "k", "v", "gate")}
    pooled = {name: np.full((b_count, h_count, t_count, d), np.nan, dtype=np.float32)
              for name in ("pooled_q", "pooled_k", "pooled_v")}
    bad = np.zeros((b_count, n), dtype=bool)
    wq = np.asarray(wq, dtype=np.float64)
    wk = np.asarray(wk, dtype=np.float64)
    heads = range(h_count) if heads is None else heads
    for b in range(b_count):
        srcs = None if src_row is None else np.asarray(src_row)[b]
        rows = [gather_rows(x[b], srcs, n) for x in (q_in, k_in, v_in, g_in)]
        bad[b] = rows[0][1]
        for h in heads:
            q_o, k_o, v_o, g_o = preprocess_rows(rows[0][0][:, h], rows[1][0][:, h], rows[2][0][:, h],
                                                 rows[3][0][:, h], wq[h], wk[h], eps, cos, sin,
                                                 rope_dim, interleaved)
            for name, val in (("q", q_o), ("k", k_o), ("v", v_o), ("gate", g_o)):
                out[name][b, :, h] = val
            pooled["pooled_q"][b, h] = vo.pool_tiles(q_o[prefix:])
            pooled["pooled_k"][b, h] = vo.pool_tiles(k_o[prefix:])
            pooled["pooled_v"][b, h] = vo.pool_tiles(v_o[prefix:])
    out.update(pooled)
    out["bad"] = bad
    return out
