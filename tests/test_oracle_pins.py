"""Pins for the CPU oracle: each test ties it to something other than itself
(hand-worked values, closed forms, invariants, brute force on tiny inputs, or
torch's CPU scaled_dot_product_attention as an independent library), so that a
dropped term, a wrong sign or index or a transposed operand fails one of them.

The method is the one "UniServe: serving FastH3 at its fastest" describes in
sections "The FastH3 workload", "Fused attention preprocessing" and "Fused
output combination".
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import vsa_oracle as vo
from block_sparse_video_gb300.synthetic import make_inputs, bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    """Round a float array to bf16 values (RNE) and return them as float64."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def _inputs(b, h, lt, la, lv, seed):
    q, k, v, g = make_inputs(b, h, lt, la, lv, seed)
    return [bf16_bits(x) for x in (q, k, v, g)]


# ---------------------------------------------------------------- counts

def test_keep_count_golden_table():
    rows = []
    with open(os.path.join(GOLDEN, "keep_counts.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if line:
                rows.append((int(line[0]), float(line[1]), int(line[3])))
    assert len(rows) >= 10
    for t, frac, k in rows:
        assert vo.keep_count(t, frac) == k, (t, frac, k)


def test_tile_lengths_ragged():
    assert list(vo.tile_lengths(150)) == [64, 64, 22]
    assert list(vo.tile_lengths(128)) == [64, 64]
    assert list(vo.tile_lengths(1)) == [1]
    assert vo.video_tile_count(72500) == 1133 and vo.tile_lengths(72500)[-1] == 52


def test_widen_is_exact():
    x = np.array([1.0, -2.5, 3.140625, 1e-30, -0.0], dtype=np.float32)
    bits = bf16_bits(torch.tensor(x).to(torch.bfloat16))
    assert np.array_equal(vo.widen(bits), _bf16(x))


# ---------------------------------------------------------------- pooling

def test_pool_brute_force_ragged():
    rng = np.random.default_rng(0)
    x = _bf16(rng.standard_normal((150, 128)))
    got = vo.pool_tiles(x)
    assert got.dtype == np.float32 and got.shape == (3, 128)
    for j, (lo, hi) in enumerate([(0, 64), (64, 128), (128, 150)]):
        for d in range(0, 128, 17):
            acc = 0.0
            for r in range(lo, hi):
                acc += x[r, d]
            assert got[j, d] == np.float32(acc / (hi - lo))


def test_pool_constant_tiles_exact():
    x = np.zeros((150, 128))
    x[:64] = 0.75
    x[64:128] = -3.0
    x[128:] = 1.5
    got = vo.pool_tiles(x)
    assert np.all(got[0] == 0.75) and np.all(got[1] == -3.0) and np.all(got[2] == 1.5)


def test_rows_beyond_sequence_are_ignored():
    """Rows past N (capacity padding) never enter the computation: poison them."""
    q, k, v, g = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, 20, 12, 150, 7)]
    base = vo.vsa_head(q, k, v, g, 32, 150, 0.4)
    pad = np.full((37, 128), np.nan)
    poisoned = vo.vsa_head(*(np.concatenate([a, pad]) for a in (q, k, v, g)), 32, 150, 0.4)
    for key in ("pooled_q", "pooled_k", "pooled_v", "scores", "index", "coarse", "out"):
        assert np.array_equal(base[key], poisoned[key]), key


# ---------------------------------------------------------------- scores / selection

def test_scores_brute_force_not_transposed():
    q, k, v, g = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, 8, 8, 200, 3)]
    r = vo.vsa_head(q, k, v, g, 16, 200, 0.2, video_tiles=[], prefix_rows=[])
    bounds = [(0, 64), (64, 128), (128, 192), (192, 200)]

    def mean(x, lo, hi, d):
        s = 0.0
        for i in range(lo, hi):
            s += x[16 + i, d]
        return np.float32(s / (hi - lo))

    qp = [[mean(q, lo, hi, d) for d in range(128)] for lo, hi in bounds]
    kp = [[mean(k, lo, hi, d) for d in range(128)] for lo, hi in bounds]
    for t in range(4):
        for j in range(4):
            dot = 0.0
            for d in range(128):
                dot += float(qp[t][d]) * float(kp[j][d])
            assert r["scores"][t, j] == pytest.approx(dot / math.sqrt(128), rel=1e-6, abs=1e-7)
    assert abs(r["scores"][1, 2] - r["scores"][2, 1]) > 1e-3  # the case is not symmetric


def test_k1_selects_argmax_brute_force():
    q, k, v, g = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, 0, 0, 640, 11)]
    r = vo.vsa_head(q, k, v, g, 0, 640, 0.01, video_tiles=[], prefix_rows=[])
    assert r["k"] == 1 and r["index"].shape == (10, 1)
    for t in range(10):
        qm = q[64 * t: 64 * t + 64].mean(axis=0)
        best, best_j = -np.inf, -1
        for j in range(10):
            km = k[64 * j: 64 * j + 64].mean(axis=0)
            s = float(np.dot(qm, km))
            if s > best:
                best, best_j = s, j
        assert r["index"][t, 0] == best_j


def test_keep_all_selects_every_tile():
    q, k, v, g = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, 4, 4, 300, 5)]
    r = vo.vsa_head(q, k, v, g, 8, 300, 1.0, video_tiles=[], prefix_rows=[])
    assert np.array_equal(r["index"], np.tile(np.arange(5), (5, 1)))


def test_select_ties_go_to_lower_index_and_output_is_ascending():
    s = np.array([1.0, 3.0, 3.0, 2.0, 3.0, -1.0], dtype=np.float32)
    assert list(vo.select_tiles(s, 1)) == [1]
    assert list(vo.select_tiles(s, 2)) == [1, 2]
    assert list(vo.select_tiles(s, 3)) == [1, 2, 4]
    assert list(vo.select_tiles(s, 4)) == [1, 2, 3, 4]
    z = np.array([0.0, -0.0, 0.0, -1.0], dtype=np.float32)  # +0 and -0 are the same score
    assert list(vo.select_tiles(z, 2)) == [0, 1]


def test_duplicate_key_tiles_tie_to_lower_index():
    q, k, v, g = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, 0, 0, 512, 9)]
    k[64 * 5: 64 * 6] = k[64 * 2: 64 * 3]  # tiles 2 and 5 score identically
    r = vo.vsa_head(q, k, v, g, 0, 512, 0.01, video_tiles=[], prefix_rows=[])
    s = r["scores"]
    assert np.array_equal(s[:, 2], s[:, 5])
    # make tile 2/5 the winner for query tile 0 by boosting its pooled query
    q[0:64] = k[64 * 2: 64 * 3] * 4.0
    r = vo.vsa_head(q, k, v, g, 0, 512, 0.01, video_tiles=[], prefix_rows=[])
    assert r["scores"][0, 2] == r["scores"][0, 5] == r["scores"][0].max()
    assert r["index"][0, 0] == 2


def test_tile_permutation_equivariance():
    lt, la, lv = 16, 16, 512
    arrs = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, lt, la, lv, 13)]
    perm = np.random.default_rng(1).permutation(8)  # new tile i holds old tile perm[i]
    rows = np.concatenate([np.arange(32)] + [32 + 64 * p + np.arange(64) for p in perm])
    base = vo.vsa_head(*arrs, 32, lv, 0.3)
    moved = vo.vsa_head(*(a[rows] for a in arrs), 32, lv, 0.3)
    inv = np.argsort(perm)
    for i in range(8):
        assert np.array_equal(np.sort(inv[base["index"][perm[i]]]), moved["index"][i])
        np.testing.assert_allclose(moved["coarse"][i], base["coarse"][perm[i]], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(moved["out"], base["out"][rows], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- coarse branch

def test_coarse_single_tile_is_pooled_v():
    q, k, v, g = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, 10, 0, 40, 2)]
    r = vo.vsa_head(q, k, v, g, 10, 40, 0.2)
    np.testing.assert_array_equal(r["coarse"][0], r["pooled_v"][0].astype(np.float64))


def test_coarse_constant_v():
    q, k, v, g = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, 8, 8, 300, 4)]
    u = _bf16(np.linspace(-1, 1, 128))
    v[16:] = u
    r = vo.vsa_head(q, k, v, g, 16, 300, 0.2, video_tiles=[], prefix_rows=[])
    np.testing.assert_allclose(r["coarse"], np.tile(u, (5, 1)), rtol=0, atol=1e-14)


def test_coarse_closed_form_two_tiles():
    """Two video tiles with known pooled vectors: query tile 0 = a*e0, key tile
    0 = e0, everything else 0; V tile 0 = e1, V tile 1 = e2. Then
    s = [[a/sqrt(128), 0], [0, 0]] and c0 = sig*e1 + (1-sig)*e2 with
    sig = 1/(1+exp(-a/sqrt(128))), c1 = (e1+e2)/2. The coarse softmax covers
    both tiles even though only k=1 of them is selected."""
    a = 3.0
    n = 128
    q = np.zeros((n, 128)); k = np.zeros((n, 128)); v = np.zeros((n, 128)); g = np.zeros((n, 128))
    q[:64, 0] = a
    k[:64, 0] = 1.0
    v[:64, 1] = 1.0
    v[64:, 2] = 1.0
    r = vo.vsa_head(q, k, v, g, 0, n, 0.2)
    assert r["k"] == 1
    s0 = a / math.sqrt(128)
    assert r["scores"][0, 0] == np.float32(s0) and r["scores"][1, 0] == 0.0 and r["scores"][0, 1] == 0.0
    sig = 1.0 / (1.0 + math.exp(-float(np.float32(s0))))
    assert r["coarse"][0, 1] == pytest.approx(sig, rel=1e-12)
    assert r["coarse"][0, 2] == pytest.approx(1.0 - sig, rel=1e-12)
    assert r["coarse"][1, 1] == pytest.approx(0.5) and r["coarse"][1, 2] == pytest.approx(0.5)
    assert list(r["index"][:, 0]) == [0, 0]  # tile 1 ties 0 == 0 -> lower index
    # out = fine + sigmoid(0) * c_tile(i): gate 0 -> 0.5
    np.testing.assert_allclose(r["out"][:64] - r["fine"][:64], 0.5 * np.tile(r["coarse"][0], (64, 1)), atol=1e-14)
    np.testing.assert_allclose(r["out"][64:] - r["fine"][64:], 0.5 * np.tile(r["coarse"][1], (64, 1)), atol=1e-14)


# ---------------------------------------------------------------- fine branch

def _sdpa(q, k, v, mask=None):
    qt = torch.from_numpy(q)[None, None]
    kt = torch.from_numpy(k)[None, None]
    vt = torch.from_numpy(v)[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m)[0, 0].numpy()


def test_keep_all_is_dense_attention_library():
    lt, la, lv = 40, 30, 300  # ragged prefix and ragged last tile
    q, k, v, g = [vo.widen(a[0, :, 1]) for a in _inputs(1, 2, lt, la, lv, 21)]
    r = vo.vsa_head(q, k, v, g, 70, lv, 1.0)
    np.testing.assert_allclose(r["fine"], _sdpa(q, k, v), rtol=1e-10, atol=1e-12)


def test_sparse_fine_matches_masked_library_attention():
    lt, la, lv = 24, 40, 700
    p = lt + la
    q, k, v, g = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, lt, la, lv, 17)]
    r = vo.vsa_head(q, k, v, g, p, lv, 0.2)
    assert r["k"] == 2
    n = p + lv
    mask = np.zeros((n, n), dtype=bool)
    mask[:p, :] = True                    # text/audio queries: every key
    mask[p:, :p] = True                   # video queries: every text/audio key
    tile_of = (np.arange(lv) // 64)
    for i in range(lv):
        sel = r["index"][tile_of[i]]
        mask[p + i, p:] = np.isin(tile_of, sel)
    np.testing.assert_allclose(r["fine"], _sdpa(q, k, v, mask), rtol=1e-10, atol=1e-12)


def test_single_video_tile_is_dense():
    q, k, v, g = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, 5, 6, 50, 8)]
    r = vo.vsa_head(q, k, v, g, 11, 50, 0.2)
    np.testing.assert_allclose(r["fine"], _sdpa(q, k, v), rtol=1e-10, atol=1e-12)


def test_constant_v_gives_constant_fine_and_closed_form_out():
    q, k, v, g = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, 20, 20, 300, 6)]
    u = _bf16(np.cos(np.arange(128)))
    v[:] = u
    r = vo.vsa_head(q, k, v, g, 40, 300, 0.2)
    np.testing.assert_allclose(r["fine"], np.tile(u, (340, 1)), rtol=0, atol=1e-14)
    sig = 1.0 / (1.0 + np.exp(-g[40:]))
    np.testing.assert_allclose(r["out"][40:], u * (1.0 + sig), rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["out"][:40], np.tile(u, (40, 1)), rtol=0, atol=1e-14)


def test_key_order_does_not_matter():
    rng = np.random.default_rng(3)
    q = _bf16(rng.standard_normal((64, 128)))
    k = _bf16(rng.standard_normal((500, 128)))
    v = _bf16(rng.standard_normal((500, 128)))
    perm = rng.permutation(500)
    np.testing.assert_allclose(vo.attention(q, k[perm], v[perm]), vo.attention(q, k, v), rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- combination

def test_zero_gate_factor_gives_fine_alone():
    """A gate pre-activation of -inf makes sigmoid exactly 0: out = fine."""
    q, k, v, g = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, 32, 32, 400, 10)]
    g[:] = -np.inf
    r = vo.vsa_head(q, k, v, g, 64, 400, 0.2)
    assert np.array_equal(r["out"], r["fine"])


def test_saturated_gate_adds_coarse_of_own_tile():
    q, k, v, g = [vo.widen(a[0, :, 0]) for a in _inputs(1, 1, 32, 32, 400, 12)]
    g[:] = 1e4
    r = vo.vsa_head(q, k, v, g, 64, 400, 0.2)
    tile_of = np.arange(400) // 64
    np.testing.assert_allclose(r["out"][64:] - r["fine"][64:], r["coarse"][tile_of], rtol=0, atol=1e-12)
    assert np.array_equal(r["out"][:64], r["fine"][:64])  # prefix rows: no coarse term
