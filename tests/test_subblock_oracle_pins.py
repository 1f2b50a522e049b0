"""Pins for the SubBlock router oracle (the SGLang Diffusion benchmark page (MiniMax-H3 on 8x H200),
section "How SubBlock Sparse Attention Works"). Each test ties the
oracle to something other than itself:
* a hand-worked budget table;
* brute-force sub-block means;
* the exact softmax mass by brute force over token pairs, when Q and K are
  constant on each sub-block (the estimate is then exact);
* the argmax of the brute-force mass;
* torch's CPU scaled_dot_product_attention at sparsity 0 and with a block mask.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import subblock_oracle as so
from oracle import vsa_oracle as vo
from block_sparse_video_gb300.synthetic import make_inputs, bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_keep_count_golden_table():
    rows = []
    with open(os.path.join(GOLDEN, "subblock_keep_counts.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if line:
                rows.append((int(line[0]), float(line[1]), int(line[4])))
    assert len(rows) >= 10
    for t, s, k in rows:
        assert so.keep_count(t, s) == k, (t, s, k)


def test_sub_counts_and_pool_brute_force_ragged():
    assert list(so.sub_counts(150)) == [16, 16, 16, 16, 16, 16, 16, 16, 16, 6, 0, 0]
    rng = np.random.default_rng(0)
    x = rng.standard_normal((150, 128)).astype(np.float32).astype(np.float64)
    got = so.sub_pool(x)
    assert got.shape == (12, 128) and got.dtype == np.float32
    for s, (lo, hi) in enumerate([(16 * i, min(16 * i + 16, 150)) for i in range(12)]):
        for d in (0, 63, 127):
            if lo >= hi:
                assert got[s, d] == 0.0
                continue
            acc = 0.0
            for r in range(lo, hi):
                acc += x[r, d]
            assert got[s, d] == np.float32(acc / (hi - lo))


def _piecewise_constant(lv, seed):
    """Q and K rows constant on every 16-token sub-block (so the mass estimate is exact)."""
    rng = np.random.default_rng(seed)
    n_sub = len(so.sub_counts(lv))
    qv = rng.standard_normal((n_sub, 128)) * 0.6
    kv = rng.standard_normal((n_sub, 128)) * 0.6
    q = np.repeat(qv, 16, axis=0)[:lv]
    k = np.repeat(kv, 16, axis=0)[:lv]
    return q, k


def test_scores_equal_log_of_the_exact_mass_on_piecewise_constant_inputs():
    lv = 64 * 3 + 37  # ragged last block: sub-blocks of 16, 16, 5 and 0 tokens
    q, k = _piecewise_constant(lv, 1)
    n_sub = so.sub_counts(lv)
    s = so.block_scores(so.sub_pool(q), so.sub_pool(k), n_sub)
    t = vo.video_tile_count(lv)
    assert s.shape == (t, t)
    for i in range(t):
        for j in range(t):
            qi = q[64 * i: min(64 * i + 64, lv)]
            kj = k[64 * j: min(64 * j + 64, lv)]
            mass = 0.0
            for r in range(qi.shape[0]):          # every token pair, no pooling
                mass += np.exp((kj @ qi[r]) / math.sqrt(128.0)).sum()
            assert s[i, j] == pytest.approx(math.log(mass), rel=2e-6, abs=2e-6), (i, j)


def test_score_is_symmetric_in_the_sub_block_order():
    rng = np.random.default_rng(2)
    qs = rng.standard_normal((8, 128)).astype(np.float32)
    ks = rng.standard_normal((8, 128)).astype(np.float32)
    n = np.full(8, 16)
    base = so.block_scores(qs, ks, n)
    perm = np.array([2, 0, 3, 1, 5, 7, 4, 6])   # shuffles sub-blocks within each block
    assert np.array_equal(so.block_scores(qs[perm], ks[perm], n), base)
    # not symmetric between query and key roles
    assert not np.allclose(so.block_scores(ks, qs, n), base)


def _inputs(b, h, lt, la, lv, seed):
    q, k, v, g = make_inputs(b, h, lt, la, lv, seed)
    return [vo.widen(bf16_bits(x))[0, :, 0] for x in (q, k, v)]


def test_budget_one_block_picks_the_largest_exact_mass():
    lv = 64 * 9
    q, k = _piecewise_constant(lv, 3)
    v = np.random.default_rng(4).standard_normal((lv, 128))
    r = so.subblock_head(q, k, v, 0, lv, 0.95, video_tiles=[], prefix_rows=[])
    assert r["k"] == 8
    for i in range(9):
        masses = []
        for j in range(9):
            qi, kj = q[64 * i: 64 * i + 64], k[64 * j: 64 * j + 64]
            masses.append(np.exp((qi @ kj.T) / math.sqrt(128.0)).sum())
        order = np.argsort(-np.array(masses), kind="stable")
        assert set(r["index"][i]) == set(order[:8]), i


def test_sparsity_zero_is_dense_attention():
    lt, la, lv = 20, 12, 64 * 4 + 9
    q, k, v = _inputs(1, 1, lt, la, lv, 5)
    r = so.subblock_head(q, k, v, lt + la, lv, 0.0)
    assert r["k"] == 5 and np.array_equal(r["index"], np.tile(np.arange(5), (5, 1)))
    tq, tk, tv = (torch.from_numpy(x[None, None]) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=1 / math.sqrt(128))[0, 0].numpy()
    assert np.allclose(r["out"], ref, atol=1e-10, rtol=1e-10)


def test_routed_output_matches_a_block_masked_sdpa():
    lt, la, lv = 30, 34, 64 * 20
    q, k, v = _inputs(1, 1, lt, la, lv, 6)
    p = lt + la
    r = so.subblock_head(q, k, v, p, lv, 0.75)
    assert r["k"] == 8
    n = p + lv
    mask = np.zeros((n, n), dtype=bool)
    mask[:p, :] = True                      # prefix queries: every key
    mask[:, :p] = True                      # every query: the prefix keys
    for t in range(20):
        for j in r["index"][t]:
            mask[p + 64 * t: p + 64 * t + 64, p + 64 * j: p + 64 * j + 64] = True
    tq, tk, tv = (torch.from_numpy(x[None, None]) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(mask),
                                                           scale=1 / math.sqrt(128))[0, 0].numpy()
    assert np.allclose(r["out"], ref, atol=1e-10, rtol=1e-10)
