"""CPU oracle for the SubBlock router feeding the block-sparse fine attention.

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import or run it; the library never does.
It shares no code with the CUDA path.

What it computes follows the SGLang Diffusion benchmark page (MiniMax-H3 on 8x H200),
section "How SubBlock Sparse Attention Works":
* the sequence is cut into 64-token query and key blocks, and each block into
  four 16-token sub-blocks on both sides (n_q = n_k = 4);
* a pooling and log-sum-exp score estimates each key block's unnormalised
  softmax mass for each query block and head;
* the router keeps the highest-scoring key blocks;
* the sparsity value is the fraction of key blocks that may be dropped, and
  the budget is rounded in units of 8 blocks;
* the kept blocks' indices go to the block-sparse attention.

Readings of what the page leaves open (each is listed with its reason in the
design notes):
* Routing covers video query blocks over video key blocks. Text and audio
  stay dense, as in the VSA fine pass (the same block-sparse attention), and
  there is no coarse branch and no gate.
* Sub-block pooling is the mean of the sub-block's valid tokens. A sub-block
  past the end of a ragged last block is empty.
* Mass estimate: each pair of sub-blocks (a of query block i, b of key block
  j) stands for n_a * n_b token pairs at logit q_a . k_b / sqrt(128), so
  score(i, j) = log sum over non-empty (a, b) of n_a n_b exp(q_a . k_b / sqrt(128)).
  This is exact when Q and K are constant on every sub-block.
* Budget: at most floor(s T) of the T key blocks are dropped (IEEE double),
  and the kept count is rounded up to a multiple of 8:
  k = min(T, 8 ceil((T - floor(s T)) / 8)).
* Ranking as in the VSA selection: scores rounded to fp32, the k highest,
  ties to the lower block index, stored ascending.
Arithmetic is fp64 except for the fp32 pooled values and scores.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import vsa_oracle as vo

SUB = 16          # tokens per sub-block
SUBS = 4          # sub-blocks per 64-token block (n_q = n_k = 4)


def keep_count(n_blocks: int, sparsity: float) -> int:
    """Kept key blocks for `sparsity` (the fraction that may be dropped), in
    units of 8 blocks: min(T, 8 * ceil((T - floor(s * T)) / 8))."""
    t = int(n_blocks)
    dropped = int(math.floor(float(sparsity) * float(t)))
    need = t - dropped
    return min(t, 8 * (-(-need // 8)))


def sub_counts(len_video: int) -> np.ndarray:
    """n for each of the 4T sub-blocks: 16, except within a ragged last block."""
    t = vo.video_tile_count(len_video)
    starts = SUB * np.arange(SUBS * t)
    return np.clip(int(len_video) - starts, 0, SUB)


def sub_pool(x_video: np.ndarray) -> np.ndarray:
    """fp32 [4T, 128]: the mean of each 16-token sub-block over its valid tokens
    (0 for an empty sub-block). The sum is taken in fp64."""
    lv = x_video.shape[0]
    n = sub_counts(lv)
    out = np.zeros((len(n), x_video.shape[1]), dtype=np.float32)
    for s, ns in enumerate(n):
        if ns:
            rows = x_video[SUB * s: SUB * s + ns]
            out[s] = (rows.sum(axis=0, dtype=np.float64) / float(ns)).astype(np.float32)
    return out


def block_scores(q_sub: np.ndarray, k_sub: np.ndarray, n_sub: np.ndarray) -> np.ndarray:
    """fp32 [T, T] estimated log softmax mass of key block j for query block i:
    log sum_{a, b} n_a n_b exp(q_sub[4i + a] . k_sub[4j + b] / sqrt(128)) over
    non-empty sub-blocks, in fp64 (a log-sum-exp), rounded to fp32."""
    t = len(n_sub) // SUBS
    logits = (q_sub.astype(np.float64) @ k_sub.astype(np.float64).T) * vo.SCALE   # [4T, 4T]
    with np.errstate(divide="ignore"):
        ln_n = np.log(n_sub.astype(np.float64))                                     # -inf when empty
    x = logits + ln_n[:, None] + ln_n[None, :]
    x = x.reshape(t, SUBS, t, SUBS).transpose(0, 2, 1, 3).reshape(t, t, SUBS * SUBS)
    m = x.max(axis=2, keepdims=True)
    lse = m[..., 0] + np.log(np.exp(x - m).sum(axis=2))
    return lse.astype(np.float32)


def subblock_head(q, k, v, prefix: int, len_video: int, sparsity: float,
                  video_tiles=None, prefix_rows=None, index_override=None):
    """SubBlock-routed attention for one (batch, head) slice: sub-block pooling
    and block scores of the video rows, top-k key blocks per video query block,
    then the fine attention over the prefix plus the kept blocks (video rows)
    or over every key (prefix rows). There is no coarse term.

    Returns the sub-pooled Q/K, block scores, the selection, and ``out`` [N, 128]
    (NaN on rows that were not requested).
    """
    q, k, v = vo.widen(q), vo.widen(k), vo.widen(v)
    n_tok = prefix + len_video
    q, k, v = q[:n_tok], k[:n_tok], v[:n_tok]
    t_count = vo.video_tile_count(len_video)
    kk = keep_count(t_count, sparsity)
    n_sub = sub_counts(len_video)
    qs = sub_pool(q[prefix:])
    ks = sub_pool(k[prefix:])
    scores = block_scores(qs, ks, n_sub)
    index = np.stack([vo.select_tiles(scores[t], kk) for t in range(t_count)])
    n = vo.tile_lengths(len_video)
    out = np.full((n_tok, q.shape[1]), np.nan)
    for t in (range(t_count) if video_tiles is None else video_tiles):
        t = int(t)
        sel = index[t]
        if index_override is not None and t in index_override:
            sel = np.asarray(index_override[t])
        rows = np.arange(prefix + t * vo.TILE, prefix + t * vo.TILE + int(n[t]))
        keys = vo.video_key_rows(prefix, len_video, sel)
        out[rows] = vo.attention(q[rows], k[keys], v[keys])
    rows_p = np.arange(prefix) if prefix_rows is None else np.asarray(prefix_rows, dtype=np.int64)
    for c in range(0, len(rows_p), vo.TILE):
        rows = rows_p[c:c + vo.TILE]
        out[rows] = vo.attention(q[rows], k, v)
    return dict(sub_q=qs, sub_k=ks, scores=scores, index=index, out=out, k=kk, n_tiles=t_count)
