"""A CPU model of the fine kernel's fast softmax arithmetic, checked against an
fp64 softmax: the numeric window in which the fast pass's fixed reference is
exact to the output tolerance, and the checks that send a row elsewhere.

The model follows the kernel's fast path, not the oracle:
  * scores t in log2 units (score * log2(e) / sqrt(128)), reference fixed at 0;
  * P = 2^t in fp32, rounded to bf16 for the P.V product, accumulated in fp32;
  * each lane's partial row sum in fp32, over its own keys (key lane l takes
    keys l, l + 128, l + 256, ...);
  * the row is kept when every lane's partial lies in [2^-60, 2^64).
It pins the window stated for the fast pass: scores within [-60, +54] in log2
units always pass, and with them the result matches the fp64 softmax within the
output tolerance; a row far outside fails a check.
"""
import numpy as np
import pytest

FLOOR = 2.0 ** -60
CEIL = 2.0 ** 64
LANES = 128


def bf16_round(x):
    """fp32 -> bf16 -> fp32, round to nearest even (finite inputs)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def fast_row(t, v):
    """t: log2-unit scores [n] (fp32), v: values [n, d]. Returns (out, kept)."""
    t = t.astype(np.float32)
    p = np.exp2(t).astype(np.float32)
    n = len(t)
    pad = (-n) % LANES
    lanes = np.concatenate([p, np.zeros(pad, np.float32)]).reshape(-1, LANES)
    partial = lanes.sum(axis=0, dtype=np.float32)
    valid = np.arange(LANES) < n  # lanes with at least one key
    kept = bool(np.all((partial[valid] >= FLOOR) & (partial[valid] < CEIL)))
    l = partial.sum(dtype=np.float32)
    o = (bf16_round(p)[:, None].astype(np.float32) * v.astype(np.float32)).sum(axis=0, dtype=np.float32)
    return o / l, kept


def exact_row(t, v):
    t = t.astype(np.float64)
    w = np.exp2(t - t.max())
    return (w[:, None] * v).sum(axis=0) / w.sum()


@pytest.mark.parametrize("center", [-50.0, -30.0, 0.0, 20.0, 45.0])
@pytest.mark.parametrize("n", [16_576, 74_624])  # a video row and a prefix row at the 10 s shape
def test_window_rows_stay_fast_and_match(center, n):
    rng = np.random.default_rng(int(center * 10) + n + 1000)
    d = 16
    errs = []
    for _ in range(3):
        t = np.clip(center + rng.normal(0.0, 3.0, n), -60.0, 54.0)
        v = rng.normal(0.0, 1.0, (n, d))
        out, kept = fast_row(t, v)
        assert kept, (center, n)
        errs.append(np.abs(out - exact_row(t, v)))
    e = np.concatenate(errs)
    assert e.max() <= 2e-2 and e.mean() <= 2e-3, (center, e.max(), e.mean())


def test_every_score_at_the_top_of_the_window_stays_fast():
    """583 keys a lane (a 74,624-key prefix row), every score at +54: each
    partial is 583 * 2^54 < 2^64."""
    n = 74_624
    t = np.full(n, 54.0)
    rng = np.random.default_rng(4)
    v = rng.normal(0.0, 1.0, (n, 8))
    out, kept = fast_row(t, v)
    assert kept
    assert np.abs(out - exact_row(t, v)).max() <= 2e-2


def test_scores_past_the_ceiling_are_sent_to_the_exact_pass():
    rng = np.random.default_rng(1)
    t = rng.normal(0.0, 1.0, 260)
    t[7] = 70.0  # one P = 2^70 leaves its lane's partial above 2^64
    _, kept = fast_row(t, rng.normal(size=(260, 16)))
    assert not kept


def test_scores_under_the_floor_are_sent_to_the_exact_pass():
    rng = np.random.default_rng(2)
    t = -80.0 + rng.normal(0.0, 1.0, 260)  # every P near 2^-80: every partial under 2^-60
    _, kept = fast_row(t, rng.normal(size=(260, 16)))
    assert not kept


def test_one_lane_far_below_the_rest_costs_a_redo_only():
    """A lane whose own keys all score far below the row's other keys fails the
    floor alone (a conservative check): the row is redone, never kept wrong."""
    rng = np.random.default_rng(3)
    t = rng.normal(0.0, 1.0, 256)
    t[5::LANES] = -90.0  # lane 5's two keys
    _, kept = fast_row(t, rng.normal(size=(256, 16)))
    assert not kept
