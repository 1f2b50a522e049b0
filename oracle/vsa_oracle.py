"""CPU oracle for the video sparse attention (VSA) forward.

TEST INFRASTRUCTURE ONLY. This module is the correctness reference the CUDA
path is checked against. Only the test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import or run it; the library never does.
It shares no code with the CUDA path.

What it computes follows "UniServe: serving FastH3 at its fastest":

* section "The FastH3 workload": the sequence is processed in tiles of 64
  tokens; text and audio queries attend to every key; video queries attend to
  all text and audio keys plus the highest-scoring 20% of video key tiles
  (rounded to a whole number of tiles); a coarse branch attends over
  mean-pooled tiles and a gate adds its output to the fine output;
* section "Fused attention preprocessing": pooling is over the valid tokens of
  a tile and the pooled statistics are FP32;
* section "Fused output combination": O_i = O_i^fine + G_i * O^coarse_tile(i);
* section "Benchmarks / Setup": the top-k tiles are selected exactly.

Conventions the page leaves open, as read here (each is listed with its reason
in the design notes): video tokens are tile-contiguous and follow the text and
audio prefix in memory; the ranking score is the scaled dot product of the
mean-pooled Q tile with the mean-pooled K tile; k = max(1, min(T, floor(f*T +
1/2))) in IEEE double; equal scores go to the lower tile index; the coarse
softmax runs over all T video tiles; a ragged last tile is pooled over its
valid tokens and only those are keys; prefix rows get no coarse term;
G = sigmoid(gate) per channel; softmax scale 1/sqrt(128).

Precision: inputs are bf16 and are widened exactly. Pooled statistics are
stored in fp32 (the page fixes that) and tile scores are rounded to fp32
before ranking, because the ranking is an integer decision and both sides must
take it in the same precision (the kernel's fp32). Everything else is fp64.

Every function is plain: a library matmul, sum or sort is the only help it
takes, with no blocking or reordering beyond row-independent chunking.
"""
from __future__ import annotations

import math

import numpy as np

TILE = 64
HEAD_DIM = 128
SCALE = 1.0 / math.sqrt(HEAD_DIM)


# ----------------------------------------------------------------------------
# Shapes and counts
# ----------------------------------------------------------------------------

def video_tile_count(len_video: int) -> int:
    """T = number of 64-token video tiles, the last one possibly ragged
    ("The FastH3 workload": VSA operates on tiles of 64 tokens)."""
    return -(-int(len_video) // TILE)


def tile_lengths(len_video: int) -> np.ndarray:
    """n_j: valid tokens of video tile j (64 except a ragged last tile)."""
    t = video_tile_count(len_video)
    n = np.full(t, TILE, dtype=np.int64)
    if t and len_video % TILE:
        n[-1] = len_video % TILE
    return n


def keep_count(n_tiles: int, keep: float) -> int:
    """k: the kept fraction of video key tiles "rounded to a whole number of
    tiles" ("The FastH3 workload"), read as round-half-up in IEEE double and
    clamped to [1, T]."""
    k = int(math.floor(float(keep) * float(n_tiles) + 0.5))
    return max(1, min(int(n_tiles), k))


# ----------------------------------------------------------------------------
# Input widening
# ----------------------------------------------------------------------------

def widen(x) -> np.ndarray:
    """bf16 values -> float64, exactly. Accepts raw bf16 bit patterns (uint16 or
    int16 arrays) or any float array that already holds the values."""
    a = np.asarray(x)
    if a.dtype in (np.uint16, np.int16):
        bits = a.view(np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# ----------------------------------------------------------------------------
# The method, one (batch, head) slice at a time. Arrays are [tokens, 128].
# ----------------------------------------------------------------------------

def pool_tiles(x_video: np.ndarray) -> np.ndarray:
    """Mean of each video tile over its valid tokens, stored as fp32
    ("Fused attention preprocessing": tile pooling over valid tokens, FP32
    pooled statistics). The sum is taken in fp64."""
    lv = x_video.shape[0]
    n = tile_lengths(lv)
    out = np.empty((len(n), x_video.shape[1]), dtype=np.float32)
    for j, nj in enumerate(n):
        rows = x_video[j * TILE: j * TILE + nj]
        out[j] = (rows.sum(axis=0, dtype=np.float64) / float(nj)).astype(np.float32)
    return out


def tile_scores(q_pooled: np.ndarray, k_pooled: np.ndarray) -> np.ndarray:
    """s[t, j] = (q_pooled[t] . k_pooled[j]) / sqrt(128): every pooled query tile
    against every pooled video key tile. Dot product in fp64, result rounded to
    fp32 (the precision the ranking is decided in)."""
    s = (q_pooled.astype(np.float64) @ k_pooled.astype(np.float64).T) * SCALE
    return s.astype(np.float32)


def select_tiles(scores_row: np.ndarray, k: int) -> np.ndarray:
    """The k highest-scoring video key tiles of one query tile, ties to the lower
    tile index, returned in ascending tile order ("The FastH3 workload": the
    highest-scoring 20% of tiles; "Benchmarks / Setup": selected exactly).
    A full sort is the brute force."""
    s = np.asarray(scores_row, dtype=np.float32)
    idx = np.arange(s.shape[0])
    order = np.lexsort((idx, -s.astype(np.float64)))  # primary: score desc; secondary: index asc
    return np.sort(order[:k])


def coarse_output(scores_row: np.ndarray, v_pooled: np.ndarray) -> np.ndarray:
    """Coarse branch for one query tile: softmax over all T video tiles of the
    tile scores, applied to the pooled V tiles ("The FastH3 workload": a second,
    coarse branch attends over mean-pooled tiles)."""
    s = np.asarray(scores_row, dtype=np.float64)
    e = np.exp(s - s.max())
    p = e / e.sum()
    return p @ v_pooled.astype(np.float64)


def attention(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray) -> np.ndarray:
    """Textbook softmax attention with scale 1/sqrt(128), two passes (max, then
    normalised exponentials), in fp64."""
    s = (q_rows @ keys.T) * SCALE
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return (e @ values) / e.sum(axis=1, keepdims=True)


def sigmoid(g: np.ndarray) -> np.ndarray:
    """The gate G = sigmoid(gate), with sigmoid(-inf) = 0 exactly."""
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-g))


def video_key_rows(prefix: int, len_video: int, tiles) -> np.ndarray:
    """Token rows a video query of a tile with selection ``tiles`` attends to:
    every text/audio row, then the valid rows of each selected video tile."""
    n = tile_lengths(len_video)
    parts = [np.arange(prefix, dtype=np.int64)]
    for j in tiles:
        start = prefix + int(j) * TILE
        parts.append(np.arange(start, start + int(n[j]), dtype=np.int64))
    return np.concatenate(parts)


def vsa_head(q, k, v, gate, prefix: int, len_video: int, keep: float,
             video_tiles=None, prefix_rows=None, index_override=None):
    """VSA forward for one (batch, head) slice.

    q, k, v, gate: [prefix + len_video, 128] (bf16 values; widened here).
    video_tiles:   query tiles whose fine/out rows to compute (default: all).
    prefix_rows:   prefix query rows to compute (default: all).
    index_override: {tile: selection} replaces the oracle's own selection for
                    those tiles in the fine branch (used when several index
                    sets are correct because of near-ties).

    Returns a dict with the pooled statistics, tile scores, selection, coarse
    output, and ``fine`` / ``out`` arrays of shape [N, 128] (NaN on rows that
    were not requested).
    """
    q = widen(q)
    k = widen(k)
    v = widen(v)
    gate = widen(gate)
    n_tok = prefix + len_video
    assert q.shape[0] >= n_tok and len_video >= 1 and prefix >= 0
    q, k, v, gate = q[:n_tok], k[:n_tok], v[:n_tok], gate[:n_tok]
    t_count = video_tile_count(len_video)
    kk = keep_count(t_count, keep)
    n = tile_lengths(len_video)

    qp = pool_tiles(q[prefix:])
    kp = pool_tiles(k[prefix:])
    vp = pool_tiles(v[prefix:])
    scores = tile_scores(qp, kp)
    index = np.stack([select_tiles(scores[t], kk) for t in range(t_count)])
    coarse = np.stack([coarse_output(scores[t], vp) for t in range(t_count)])

    fine = np.full((n_tok, q.shape[1]), np.nan)
    out = np.full((n_tok, q.shape[1]), np.nan)
    if video_tiles is None:
        video_tiles = range(t_count)
    for t in video_tiles:
        t = int(t)
        sel = index[t]
        if index_override is not None and t in index_override:
            sel = np.asarray(index_override[t])
        rows = np.arange(prefix + t * TILE, prefix + t * TILE + int(n[t]))
        keys = video_key_rows(prefix, len_video, sel)
        o = attention(q[rows], k[keys], v[keys])
        fine[rows] = o
        out[rows] = o + sigmoid(gate[rows]) * coarse[t][None, :]
    if prefix_rows is None:
        prefix_rows = np.arange(prefix)
    prefix_rows = np.asarray(prefix_rows, dtype=np.int64)
    for c in range(0, len(prefix_rows), TILE):  # row-independent chunks
        rows = prefix_rows[c:c + TILE]
        o = attention(q[rows], k, v)
        fine[rows] = o
        out[rows] = o
    return dict(pooled_q=qp, pooled_k=kp, pooled_v=vp, scores=scores, index=index,
                coarse=coarse, fine=fine, out=out, k=kk, n_tiles=t_count)


def vsa_forward(q, k, v, gate, len_text: int, len_audio: int, len_video: int,
                keep: float, heads=None, batches=None, **kw):
    """VSA forward over [B, N, H, 128] inputs, one (b, h) slice at a time.
    Returns {(b, h): vsa_head(...) result}."""
    prefix = int(len_text) + int(len_audio)
    b_count, _, h_count, _ = np.asarray(q).shape
    res = {}
    for b in (range(b_count) if batches is None else batches):
        for h in (range(h_count) if heads is None else heads):
            res[(b, h)] = vsa_head(q[b, :, h], k[b, :, h], v[b, :, h], gate[b, :, h],
                                   prefix, len_video, keep, **kw)
    return res
