"""Plant plausible mistakes in the CPU oracle and check that its pins catch each.

Every mutation is applied with monkeypatch to the oracle module only, on the
CPU; the pins in test_oracle_pins are then run against the mutated oracle and
at least one must fail.
"""
import math

import numpy as np
import pytest

from oracle import vsa_oracle as vo
import tests.test_oracle_pins as pins

PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


def _pool_divide_by_64(x_video):
    lv = x_video.shape[0]
    n = vo.tile_lengths(lv)
    out = np.empty((len(n), x_video.shape[1]), dtype=np.float32)
    for j, nj in enumerate(n):
        out[j] = (x_video[j * 64: j * 64 + nj].sum(axis=0) / 64.0).astype(np.float32)
    return out


def _scores_transposed(qp, kp):
    return ((kp.astype(np.float64) @ qp.astype(np.float64).T) * vo.SCALE).astype(np.float32)


def _scores_no_scale(qp, kp):
    return (qp.astype(np.float64) @ kp.astype(np.float64).T).astype(np.float32)


def _select_ties_high(row, k):
    s = np.asarray(row, dtype=np.float64)
    idx = np.arange(s.shape[0])
    return np.sort(np.lexsort((-idx, -s))[:k])


def _select_unsorted(row, k):
    s = np.asarray(row, dtype=np.float64)
    return np.lexsort((np.arange(s.shape[0]), -s))[:k]


def _coarse_wrong_sign(row, vp):
    s = np.asarray(row, dtype=np.float64)
    e = np.exp(-(s - s.min()))
    return (e / e.sum()) @ vp.astype(np.float64)


def _attention_no_scale(q, k, v):
    s = q @ k.T
    e = np.exp(s - s.max(axis=1, keepdims=True))
    return (e @ v) / e.sum(axis=1, keepdims=True)


def _sigmoid_flipped(g):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(g))


def _keys_without_prefix(prefix, lv, tiles):
    n = vo.tile_lengths(lv)
    return np.concatenate([prefix + j * 64 + np.arange(n[j]) for j in tiles])


def _keep_truncates(t, f):
    return max(1, min(t, int(f * t)))


MUTATIONS = {
    "pool divides by 64 on the ragged tile": ("pool_tiles", _pool_divide_by_64),
    "tile scores transposed": ("tile_scores", _scores_transposed),
    "tile scores unscaled": ("tile_scores", _scores_no_scale),
    "ties go to the higher index": ("select_tiles", _select_ties_high),
    "selection not ascending": ("select_tiles", _select_unsorted),
    "coarse softmax sign flipped": ("coarse_output", _coarse_wrong_sign),
    "fine attention unscaled": ("attention", _attention_no_scale),
    "gate sigmoid sign flipped": ("sigmoid", _sigmoid_flipped),
    "video queries miss the prefix keys": ("video_key_rows", _keys_without_prefix),
    "k truncated instead of rounded": ("keep_count", _keep_truncates),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(vo, attr, fn)
    caught = []
    for t in PIN_TESTS:
        try:
            t()
        except Exception:  # an assertion, or a shape error the mistake causes
            caught.append(t.__name__)
    assert caught, f"no pin caught: {name}"
