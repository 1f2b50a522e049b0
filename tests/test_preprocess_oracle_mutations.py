"""Plant plausible mistakes in the preprocessing oracle and check that its pins
catch each. Mutations are applied with monkeypatch to the oracle module only,
on the CPU."""
import numpy as np
import pytest

from oracle import preprocess_oracle as po
import tests.test_preprocess_oracle_pins as pins

PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]
_rope = po.rope
_round = po.round_bf16


def _norm_no_eps(x, w, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True)) * np.asarray(w, dtype=np.float64)


def _norm_sum_not_mean(x, w, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt((x * x).sum(axis=-1, keepdims=True) + eps) * np.asarray(w, dtype=np.float64)


def _norm_no_weight(x, w, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)


def _rope_backwards(x, cos, sin, rope_dim, interleaved):
    return _rope(x, cos, -np.asarray(sin), rope_dim, interleaved)


def _rope_reflection(x, cos, sin, rope_dim, interleaved):
    x = np.array(x, dtype=np.float64)
    if rope_dim == 0:
        return x
    a_idx, b_idx = po.rope_pairs(rope_dim, interleaved)
    a, b = x[..., a_idx].copy(), x[..., b_idx].copy()
    x[..., a_idx] = a * cos + b * sin
    x[..., b_idx] = a * sin - b * cos
    return x


def _rope_layout_ignored(x, cos, sin, rope_dim, interleaved):
    return _rope(x, cos, sin, rope_dim, True)


def _pairs_off_by_one(rope_dim, interleaved):
    half = rope_dim // 2
    i = np.arange(half)
    if interleaved:
        return 2 * i, 2 * i + 1
    return i, (i + half + 1) % rope_dim


def _rows_no_intermediate_rounding(q, k, v, gate, wq, wk, eps, cos, sin, rope_dim, interleaved):
    q_out = _round(_rope(po.rms_norm(q, wq, eps), cos, sin, rope_dim, interleaved))
    k_out = _round(_rope(po.rms_norm(k, wk, eps), cos, sin, rope_dim, interleaved))
    return q_out, k_out, np.array(v, dtype=np.float64), np.array(gate, dtype=np.float64)


def _round_truncates(x):
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    step = np.ldexp(1.0, np.maximum(e, -125) - 8)
    return np.trunc(x / step) * step


def _gather_clamps(proj, src_row, n_rows):
    proj = np.asarray(proj)
    src = np.arange(n_rows) if src_row is None else np.asarray(src_row, dtype=np.int64)
    bad = (src < 0) | (src >= proj.shape[0])
    return proj[np.clip(src, 0, proj.shape[0] - 1)].astype(np.float64), bad


def _rows_gate_is_v(q, k, v, gate, wq, wk, eps, cos, sin, rope_dim, interleaved):
    q_out, k_out, v_out, _ = _rows(q, k, v, gate, wq, wk, eps, cos, sin, rope_dim, interleaved)
    return q_out, k_out, v_out, v_out.copy()


_rows = po.preprocess_rows

MUTATIONS = {
    "RMSNorm without eps": ("rms_norm", _norm_no_eps),
    "RMSNorm over the sum of squares": ("rms_norm", _norm_sum_not_mean),
    "RMSNorm weight dropped": ("rms_norm", _norm_no_weight),
    "RoPE rotates backwards": ("rope", _rope_backwards),
    "RoPE reflects instead of rotating": ("rope", _rope_reflection),
    "RoPE half-split layout treated as interleaved": ("rope", _rope_layout_ignored),
    "RoPE half-split partner off by one": ("rope_pairs", _pairs_off_by_one),
    "no rounding between norm and RoPE": ("preprocess_rows", _rows_no_intermediate_rounding),
    "bf16 rounding truncates": ("round_bf16", _round_truncates),
    "out-of-range rows clamped instead of zeroed": ("gather_rows", _gather_clamps),
    "gate output copies V": ("preprocess_rows", _rows_gate_is_v),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(po, attr, fn)
    caught = []
    for t in PIN_TESTS:
        try:
            t()
        except Exception:  # an assertion, or a shape error the mistake causes
            caught.append(t.__name__)
    assert caught, f"no pin caught: {name}"
