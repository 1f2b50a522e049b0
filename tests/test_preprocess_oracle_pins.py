"""Pins for the preprocessing oracle ("UniServe: serving FastH3 at its fastest",
section "Fused attention preprocessing": Q/K RMSNorm, partial RoPE, pooling
over valid tokens, tile packing, gate copy).

Each test ties the oracle to something other than itself. The anchors are:
* hand-worked values (tests/golden/preprocess_norm_rope.txt);
* torch's own bf16 conversion;
* complex multiplication as an independent statement of the rotation;
* RoPE's relative-position property;
* the permutation relating the two pair layouts;
* brute-force loops.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import preprocess_oracle as po
from oracle import vsa_oracle as vo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "preprocess_norm_rope.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if line:
                rows.append((int(line[0]), float(line[1]), float(line[2]), float(line[3]), float(line[4])))
    return rows


def _row_3_4():
    x = np.zeros(128)
    x[0], x[1] = 3.0, 4.0
    return x


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_hand_worked_ties():
    r = po.round_bf16
    assert r(1.0 + 2.0 ** -8) == 1.0                       # tie, 1.0 is even
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6       # tie, rounds up to the even neighbour
    assert r(-(1.0 + 2.0 ** -8)) == -1.0
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7  # just above the tie
    assert r(3 * 2.0 ** -134) == 2.0 ** -132               # subnormal spacing 2^-133, tie to even
    assert r(255.5) == 256.0 and r(254.5) == 254.0        # spacing 1 in [128, 256), 2 in [256, 512)
    assert r(0.0) == 0.0


def test_round_bf16_matches_torch_conversion_of_fp32():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(po.round_bf16(x.astype(np.float64)), want)


# ---------------------------------------------------------------- RMSNorm

def test_rms_norm_hand_worked():
    y = po.rms_norm(_row_3_4(), np.ones(128), 25.0 / 128.0)
    assert y[0] == 4.8 and y[1] == 6.4 and np.all(y[2:] == 0.0)
    y0 = po.rms_norm(_row_3_4(), np.ones(128), 0.0)
    assert y0[0] == pytest.approx(3.0 * math.sqrt(128.0) / 5.0, rel=1e-15)


def test_rms_norm_unit_rms_rows_independent_and_weighted():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 128))
    x[1] = 10.0 * x[0]                    # a scaled copy normalises to the same row
    y = po.rms_norm(x, np.ones(128), 0.0)
    assert np.allclose((y * y).mean(axis=1), 1.0, rtol=1e-14)
    assert np.allclose(y[0], y[1], rtol=1e-14)
    w = rng.standard_normal(128)
    assert np.allclose(po.rms_norm(x, w, 0.0), y * w, rtol=1e-14)
    assert np.all(po.rms_norm(np.zeros((1, 128)), w, 1e-6) == 0.0)  # eps keeps zero rows finite


# ---------------------------------------------------------------- RoPE

def test_rope_quarter_turn_and_identity():
    x = np.zeros((2, 128))
    x[0, 0], x[1, 1] = 1.0, 1.0
    c = np.zeros((2, 1))
    s = np.ones((2, 1))
    y = po.rope(x, c, s, 2, True)
    assert y[0, 0] == 0.0 and y[0, 1] == 1.0      # (1, 0) turns to (0, 1)
    assert y[1, 0] == -1.0 and y[1, 1] == 0.0     # (0, 1) turns to (-1, 0)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 128))
    assert np.array_equal(po.rope(x, np.ones((4, 48)), np.zeros((4, 48)), 96, False), x)


def _angles(n_rows, half, seed):
    rng = np.random.default_rng(seed)
    th = rng.uniform(-math.pi, math.pi, (n_rows, half))
    return th, np.cos(th), np.sin(th)


def test_rope_is_complex_multiplication_both_layouts():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, 128))
    th, c, s = _angles(5, 48, 5)
    rot = np.exp(1j * th)
    # interleaved pairs (2i, 2i+1)
    y = po.rope(x, c, s, 96, True)
    z = (x[:, 0:96:2] + 1j * x[:, 1:96:2]) * rot
    assert np.allclose(y[:, 0:96:2], z.real, atol=1e-13) and np.allclose(y[:, 1:96:2], z.imag, atol=1e-13)
    assert np.array_equal(y[:, 96:], x[:, 96:])
    # half-split pairs (i, i + 48)
    y = po.rope(x, c, s, 96, False)
    z = (x[:, :48] + 1j * x[:, 48:96]) * rot
    assert np.allclose(y[:, :48], z.real, atol=1e-13) and np.allclose(y[:, 48:96], z.imag, atol=1e-13)
    assert np.array_equal(y[:, 96:], x[:, 96:])


def test_rope_layouts_are_a_channel_permutation_of_each_other():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 128))
    _, c, s = _angles(3, 32, 7)
    perm = np.arange(128)
    perm[0:64:2] = np.arange(32)        # interleaved slot 2i <- half-split channel i
    perm[1:64:2] = np.arange(32) + 32   # interleaved slot 2i+1 <- half-split channel i + 32
    y_half = po.rope(x, c, s, 64, False)
    y_int = po.rope(x[:, perm], c, s, 64, True)
    assert np.allclose(y_int, y_half[:, perm], atol=1e-14)


def test_rope_relative_position_property():
    """With angles linear in position, <rope(q, m), rope(k, n)> depends only on m - n."""
    rng = np.random.default_rng(8)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    omega = 10000.0 ** (-np.arange(48) / 48.0)

    def at(x, pos, inter):
        th = pos * omega
        return po.rope(x[None], np.cos(th)[None], np.sin(th)[None], 96, inter)[0]

    for inter in (True, False):
        d1 = at(q, 7.0, inter) @ at(k, 3.0, inter)
        d2 = at(q, 107.0, inter) @ at(k, 103.0, inter)
        d3 = at(q, 3.0, inter) @ at(k, 7.0, inter)
        assert abs(d1 - d2) < 1e-10 and abs(d1 - d3) > 1e-3
        pair_norms = lambda y: y[0:96:2] ** 2 + y[1:96:2] ** 2 if inter else y[:48] ** 2 + y[48:96] ** 2
        assert np.allclose(pair_norms(at(q, 11.0, inter)), pair_norms(q), rtol=1e-12)


# ---------------------------------------------------------------- the fused row work

def test_norm_round_rope_round_golden():
    rows = _golden_rows()
    assert len(rows) >= 2
    for rope_dim, c, s, o0, o1 in rows:
        half = max(rope_dim // 2, 1)
        cos = np.full((1, half), np.float32(c), dtype=np.float64)
        sin = np.full((1, half), np.float32(s), dtype=np.float64)
        x = _row_3_4()[None]
        q_out, k_out, _, _ = po.preprocess_rows(x, x, x, x, np.ones(128), np.ones(128), 25.0 / 128.0,
                                                cos[:, :rope_dim // 2], sin[:, :rope_dim // 2],
                                                rope_dim, True)
        for out in (q_out, k_out):
            assert out[0, 0] == o0 and out[0, 1] == o1 and np.all(out[0, 2:] == 0.0), (rope_dim, out[0, :2])


def test_gather_identity_permutation_and_out_of_range():
    rng = np.random.default_rng(9)
    proj = rng.standard_normal((10, 2, 128))
    rows, bad = po.gather_rows(proj, None, 7)
    assert np.array_equal(rows, proj[:7]) and not bad.any()
    src = np.array([9, 0, 4, 4, -1, 10, 2])
    rows, bad = po.gather_rows(proj, src, 7)
    assert list(bad) == [False, False, False, False, True, True, False]
    for n, j in enumerate(src):
        if 0 <= j < 10:
            assert np.array_equal(rows[n], proj[j])
        else:
            assert np.all(rows[n] == 0.0)


def _case(b, s_in, h, prefix, lv, seed):
    rng = np.random.default_rng(seed)
    def bf(shape):
        return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
    ins = [bf((b, s_in, h, 128)) for _ in range(4)]
    bits = [x.view(torch.int16).numpy().view(np.uint16) for x in ins]
    n = prefix + lv
    wq = 1.0 + 0.1 * rng.standard_normal((h, 128))
    wk = 1.0 + 0.1 * rng.standard_normal((h, 128))
    th = rng.uniform(-math.pi, math.pi, (n, 48))
    return bits, wq, wk, np.cos(th), np.sin(th)


def test_packing_reads_the_mapped_rows_and_never_the_padding():
    b, s_in, h, prefix, lv = 2, 300, 2, 70, 150
    n = prefix + lv
    bits, wq, wk, c, s = _case(b, s_in, h, prefix, lv, 10)
    rng = np.random.default_rng(11)
    src = np.stack([rng.permutation(s_in)[:n] for _ in range(b)])
    got = po.preprocess(*bits, prefix, lv, wq, wk, 1e-6, c, s, 96, True, src_row=src)
    # the same rows, moved to positions 0..n-1 of a buffer whose other rows are NaN
    packed = []
    for x in bits:
        w = vo.widen(x)
        buf = np.full((b, n + 17, h, 128), np.nan)
        for bb in range(b):
            buf[bb, :n] = w[bb, src[bb]]
        packed.append(buf)
    ref = po.preprocess(*packed, prefix, lv, wq, wk, 1e-6, c, s, 96, True)
    for key in ("q", "k", "v", "gate", "pooled_q", "pooled_k", "pooled_v"):
        assert np.array_equal(got[key], ref[key]), key
    assert not got["bad"].any()
    # V and gate are copies of the mapped rows
    for key, x in (("v", bits[2]), ("gate", bits[3])):
        w = vo.widen(x)
        for bb in range(b):
            assert np.array_equal(got[key][bb], w[bb, src[bb]])


def test_pooled_statistics_are_tile_means_of_the_video_outputs():
    b, s_in, h, prefix, lv = 1, 260, 1, 37, 150   # ragged last tile of 22 tokens
    bits, wq, wk, c, s = _case(b, s_in, h, prefix, lv, 12)
    got = po.preprocess(*bits, prefix, lv, wq, wk, 1e-6, c[: prefix + lv], s[: prefix + lv], 96, False)
    for name in ("q", "k", "v"):
        pooled = got["pooled_" + name][0, 0]
        for j, (lo, hi) in enumerate([(0, 64), (64, 128), (128, 150)]):
            for d in (0, 5, 95, 96, 127):
                acc = 0.0
                for r in range(prefix + lo, prefix + hi):
                    acc += got[name][0, r, 0, d]
                assert pooled[j, d] == np.float32(acc / (hi - lo)), (name, j, d)


def test_out_of_range_map_entries_give_zero_rows_and_are_reported():
    b, s_in, h, prefix, lv = 1, 100, 1, 10, 64
    bits, wq, wk, c, s = _case(b, s_in, h, prefix, lv, 13)
    src = np.arange(prefix + lv)[None].copy()
    src[0, 3] = 100
    src[0, 40] = -5
    got = po.preprocess(*bits, prefix, lv, wq, wk, 1e-6, c[:74], s[:74], 96, True, src_row=src)
    assert list(np.nonzero(got["bad"][0])[0]) == [3, 40]
    for key in ("q", "k", "v", "gate"):
        assert np.all(got[key][0, 3] == 0.0) and np.all(got[key][0, 40] == 0.0)
