"""Plant plausible mistakes in the SubBlock oracle and check that its pins
catch each (monkeypatch on the oracle module, CPU only)."""
import math

import numpy as np
import pytest

from oracle import subblock_oracle as so
from oracle import vsa_oracle as vo
import tests.test_subblock_oracle_pins as pins

PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]
_scores = so.block_scores


def _keep_rounds_down(t, s):
    need = t - int(math.floor(s * t))
    return max(1, min(t, 8 * (need // 8)))


def _keep_ignores_units(t, s):
    return t - int(math.floor(s * t))


def _keep_fraction_kept(t, s):
    return min(t, 8 * (-(-(t - int(math.floor((1 - s) * t))) // 8)))


def _pool_divides_by_16(x):
    n = so.sub_counts(x.shape[0])
    out = np.zeros((len(n), x.shape[1]), dtype=np.float32)
    for s, ns in enumerate(n):
        out[s] = (x[16 * s: 16 * s + ns].sum(axis=0) / 16.0).astype(np.float32)
    return out


def _scores_max_not_lse(qs, ks, n):
    t = len(n) // 4
    x = (qs.astype(np.float64) @ ks.astype(np.float64).T) * vo.SCALE
    x = x.reshape(t, 4, t, 4).transpose(0, 2, 1, 3).reshape(t, t, 16)
    return x.max(axis=2).astype(np.float32)


def _scores_no_counts(qs, ks, n):
    return _scores(qs, ks, np.where(n > 0, 16, 0))


def _scores_transposed(qs, ks, n):
    return _scores(ks, qs, n)


def _scores_unscaled(qs, ks, n):
    return _scores(qs * np.float32(math.sqrt(128.0)), ks, n)


def _scores_block_mean(qs, ks, n):
    t = len(n) // 4
    qm = qs.reshape(t, 4, -1).mean(axis=1)
    km = ks.reshape(t, 4, -1).mean(axis=1)
    return ((qm.astype(np.float64) @ km.astype(np.float64).T) * vo.SCALE).astype(np.float32)


MUTATIONS = {
    "budget rounded down": ("keep_count", _keep_rounds_down),
    "budget not in units of 8": ("keep_count", _keep_ignores_units),
    "sparsity read as the kept fraction": ("keep_count", _keep_fraction_kept),
    "sub-block mean divides by 16 on a ragged block": ("sub_pool", _pool_divides_by_16),
    "max instead of log-sum-exp": ("block_scores", _scores_max_not_lse),
    "sub-block sizes ignored": ("block_scores", _scores_no_counts),
    "query and key roles swapped": ("block_scores", _scores_transposed),
    "logits unscaled": ("block_scores", _scores_unscaled),
    "whole-block means (no sub-blocks)": ("block_scores", _scores_block_mean),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(so, attr, fn)
    caught = []
    for t in PIN_TESTS:
        try:
            t()
        except Exception:
            caught.append(t.__name__)
    assert caught, f"no pin caught: {name}"
