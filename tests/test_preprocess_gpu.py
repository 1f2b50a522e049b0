"""GPU parity of the fused attention preprocessing ("UniServe: serving FastH3 at
its fastest", section "Fused attention preprocessing") against the CPU oracle,
through the C ABI.

Tolerances, derived from the arithmetic:
* V and gate are copies: bit-exact.
* Q and K: the kernel computes in fp32 and the oracle in fp64, and each rounds
  to bf16 twice (after the norm, after RoPE). Near a rounding boundary the two
  can land one bf16 step apart at either rounding. A step is at most 2^-7 of
  the value. A step in the normalised pair (a, b) moves a rotated output by at
  most 2^-7 (|a| + |b|), and the last rounding adds one step of the output.
  So per element |gpu - oracle| <= 2^-5 (|a'| + |b'|), where (a', b') is the
  oracle's output pair (|a'| + |b'| >= (|a| + |b|) / sqrt 2). Unrotated
  channels use |y| in its place. The test also requires at least 98% of the
  elements to be bit-identical.
* Pooled statistics are checked two ways. Against the fp64 tile means of the
  kernel's own packed output, they hold to the error of a 64-term fp32 sum
  (<= 2^-18 of the mean absolute value). Against the oracle's pooled values
  they hold within the mean of the per-element bounds above.
* vsa_forward_preprocessed over the packed tensors must equal, bit for bit,
  vsa_forward over the same tensors. Both pool the same bf16 values in the same
  row order in fp32.
"""
import numpy as np
import pytest
import torch

import block_sparse_video_gb300 as bsv
from block_sparse_video_gb300.synthetic import (make_norm_weights, make_projections, make_rope_tables,
                                                make_row_map, bf16_bits)
from oracle import preprocess_oracle as po
from oracle import vsa_oracle as vo

pytestmark = pytest.mark.gpu


def _setup(b, h, lt, la, lv, rows_in, rope_dim, seed, mapped=True, device="cuda"):
    n = lt + la + lv
    proj = make_projections(b, rows_in, h, seed, device=device)
    ins = [proj[:, :, i] for i in range(4)]  # views with row stride 4 * H * 128
    wq, wk = make_norm_weights(h, seed + 1)
    cos, sin = make_rope_tables(lt, la, lv, rope_dim)
    src = make_row_map(b, n, rows_in, seed + 2) if mapped else None
    return proj, ins, wq, wk, cos, sin, src


def _gpu(op, ins, wq, wk, cos, sin, src, rope_dim, inter, eps=1e-6):
    dev = op.device
    return op.preprocess(*ins, wq.to(dev), wk.to(dev), cos.to(dev) if rope_dim else None,
                         sin.to(dev) if rope_dim else None, rope_dim, inter, eps,
                         None if src is None else src.to(dev))


def _pair_magnitude(y, rope_dim, inter):
    """|a'| + |b'| for each rotated channel's pair; |y| for the others."""
    m = np.abs(y).copy()
    if rope_dim:
        a_idx, b_idx = po.rope_pairs(rope_dim, inter)
        s = np.abs(y[..., a_idx]) + np.abs(y[..., b_idx])
        m[..., a_idx] = s
        m[..., b_idx] = s
    return m


def _check_qk(got, want, rope_dim, inter, what):
    got = np.asarray(got, dtype=np.float64)
    bound = 2.0 ** -5 * _pair_magnitude(want, rope_dim, inter) + 1e-30
    err = np.abs(got - want)
    assert np.all(err <= bound), (what, float((err / bound).max()))
    exact = np.mean(got == want)
    assert exact >= 0.98, (what, exact)
    return err


def _compare(op, out, ins_cpu, wq, wk, cos, sin, src, lt, la, lv, rope_dim, inter, eps=1e-6):
    b, h = op.batch, op.num_heads
    prefix = lt + la
    bits = [bf16_bits(x.contiguous()) for x in ins_cpu]
    ref = po.preprocess(*bits, prefix, lv, wq.numpy(), wk.numpy(), eps, cos.numpy(), sin.numpy(),
                        rope_dim, inter, src_row=None if src is None else src.numpy())
    got = [x.float().cpu().double().numpy() for x in out]
    for name, g in zip(("v", "gate"), got[2:]):
        assert np.array_equal(g, ref[name]), name
    errs = {}
    for name, g in zip(("q", "k"), got[:2]):
        errs[name] = _check_qk(g, ref[name], rope_dim, inter, name)
    views = op.debug_views()
    t = op.n_tiles
    n_j = vo.tile_lengths(lv)
    for i, name in enumerate(("q", "k", "v")):
        pooled = views["pooled_" + name].cpu().double().numpy()
        # against the tile means of the kernel's own packed output
        vid = got[i][:, prefix:]                       # [B, Lv, H, 128]
        for j in range(t):
            rows = vid[:, 64 * j: 64 * j + n_j[j]]
            mean = rows.mean(axis=1)                    # [B, H, 128]
            mabs = np.abs(rows).mean(axis=1)
            assert np.all(np.abs(pooled[:, :, j] - mean) <= 2.0 ** -18 * mabs + 1e-30), (name, j)
        # against the oracle's pooled values
        if name in errs:
            e = errs[name][:, prefix:]
            tol = np.stack([e[:, 64 * j: 64 * j + n_j[j]].mean(axis=1) for j in range(t)], axis=2)
            tol = tol + 2.0 ** -18 * np.abs(pooled) + 1e-7
            assert np.all(np.abs(pooled - ref["pooled_" + name]) <= tol), name
        else:
            assert np.allclose(pooled, ref["pooled_" + name], rtol=1e-6, atol=1e-7), name
    return ref


@pytest.mark.parametrize("inter", [True, False])
def test_preprocess_matches_oracle_mapped_capacity_buffer(cuda_ok, inter):
    # odd head count (a half-filled warp), ragged prefix tile and ragged last video tile,
    # a capacity buffer with NaN padding rows that the map never selects
    b, h, lt, la, lv = 2, 3, 37, 50, 64 * 5 + 11
    n = lt + la + lv
    rows_in = n + 100
    proj, ins, wq, wk, cos, sin, src = _setup(b, h, lt, la, lv, rows_in, 96, 21)
    used = torch.zeros((b, rows_in), dtype=torch.bool)
    for bb in range(b):
        used[bb, src[bb].long()] = True
    proj[~used.cuda()] = float("nan")
    op = bsv.VSA(b, h, lt, la, lv, 0.2)
    out = _gpu(op, ins, wq, wk, cos, sin, src, 96, inter)
    op.check()
    _compare(op, out, [x.cpu() for x in ins], wq, wk, cos, sin, src, lt, la, lv, 96, inter)


@pytest.mark.parametrize("rope_dim", [0, 16, 128])
def test_preprocess_rope_widths_identity_map(cuda_ok, rope_dim):
    b, h, lt, la, lv = 1, 8, 64, 0, 64 * 3
    n = lt + la + lv
    proj, ins, wq, wk, cos, sin, _ = _setup(b, h, lt, la, lv, n, rope_dim, 22, mapped=False)
    op = bsv.VSA(b, h, lt, la, lv, 0.3)
    out = _gpu(op, ins, wq, wk, cos, sin, None, rope_dim, rope_dim != 16)
    op.check()
    _compare(op, out, [x.cpu() for x in ins], wq, wk, cos, sin, None, lt, la, lv, rope_dim, rope_dim != 16)


def test_preprocess_separate_buffers_and_empty_prefix(cuda_ok):
    b, h, lt, la, lv = 1, 17, 0, 0, 64 * 2 + 1   # 17 heads: three CTAs of heads, the last one partial
    n = lv
    _, _, wq, wk, cos, sin, src = _setup(b, h, lt, la, lv, n + 9, 96, 23)
    ins = [make_projections(b, n + 9, h, 30 + i, device="cuda")[:, :, 0].contiguous() for i in range(4)]
    op = bsv.VSA(b, h, lt, la, lv, 0.2)
    out = _gpu(op, ins, wq, wk, cos, sin, src, 96, True)
    op.check()
    _compare(op, out, [x.cpu() for x in ins], wq, wk, cos, sin, src, lt, la, lv, 96, True)


def test_bad_map_entries_give_zero_rows_and_are_reported(cuda_ok):
    b, h, lt, la, lv = 1, 2, 10, 10, 64 * 2
    n = lt + la + lv
    rows_in = n + 5
    proj, ins, wq, wk, cos, sin, src = _setup(b, h, lt, la, lv, rows_in, 96, 24)
    src[0, 3] = rows_in
    src[0, 100] = -7
    op = bsv.VSA(b, h, lt, la, lv, 0.2)
    out = _gpu(op, ins, wq, wk, cos, sin, src, 96, True)
    with pytest.raises(bsv.VsaError) as e:
        op.check()
    assert e.value.status == bsv.VSA_ERR_INVALID_ARG
    ref = _compare(op, out, [x.cpu() for x in ins], wq, wk, cos, sin, src, lt, la, lv, 96, True)
    assert list(np.nonzero(ref["bad"][0])[0]) == [3, 100]
    for x in out:
        assert torch.count_nonzero(x[0, 3]) == 0 and torch.count_nonzero(x[0, 100]) == 0
    # the next forward over these tensors still reports it; a plain forward clears it
    op.forward_preprocessed(*out)
    with pytest.raises(bsv.VsaError):
        op.check()
    op(*out)
    op.check()


def test_fused_forward_equals_unfused_and_matches_oracle(cuda_ok):
    b, h, lt, la, lv = 1, 4, 100, 60, 64 * 12 + 5
    n = lt + la + lv
    rows_in = n + 64
    proj, ins, wq, wk, cos, sin, src = _setup(b, h, lt, la, lv, rows_in, 96, 25)
    op = bsv.VSA(b, h, lt, la, lv, 0.25)
    q, k, v, g = _gpu(op, ins, wq, wk, cos, sin, src, 96, True)
    fused = op.forward_preprocessed(q, k, v, g).clone()
    op.check()
    fused_idx = op.debug_views()["tile_index"].clone()
    plain = op(q, k, v, g)
    op.check()
    assert torch.equal(fused.view(torch.int16), plain.view(torch.int16))
    assert torch.equal(fused_idx, op.debug_views()["tile_index"])
    # the whole chain against the oracle chain (preprocess, then the forward), two heads
    bits = [bf16_bits(x.cpu()) for x in ins]
    pre = po.preprocess(*bits, lt + la, lv, wq.numpy(), wk.numpy(), 1e-6, cos.numpy(), sin.numpy(), 96, True,
                        src_row=src.numpy(), heads=[0, 3])
    got = fused.float().cpu().double().numpy()
    errs = []
    for hh in (0, 3):
        r = vo.vsa_head(pre["q"][0, :, hh], pre["k"][0, :, hh], pre["v"][0, :, hh], pre["gate"][0, :, hh],
                        lt + la, lv, 0.25)
        errs.append(np.abs(got[0, :, hh] - r["out"]))
    e = np.concatenate(errs)
    assert e.max() <= 2e-2 and e.mean() <= 2e-3, (e.max(), e.mean())


def test_preprocess_10s_shape_sampled(cuda_ok):
    """The 10 s FastH3 shape (56 heads, 1,024 + 1,024 + 72,576 tokens) from a
    78,080-row capacity buffer, the launch the benchmark times; sampled tiles
    and every head checked against the oracle."""
    b, h, lt, la, lv = 1, 56, 1024, 1024, 72576
    n = lt + la + lv
    rows_in = 78080
    proj, ins, wq, wk, cos, sin, _ = _setup(b, h, lt, la, lv, rows_in, 96, 26, mapped=False)
    op = bsv.VSA(b, h, lt, la, lv, 0.2)
    out = _gpu(op, ins, wq, wk, cos, sin, None, 96, True)
    op.check()
    views = op.debug_views()
    rng = np.random.default_rng(0)
    tiles = sorted(set(rng.choice(op.n_tiles, 6, replace=False).tolist()) | {0, op.n_tiles - 1})
    prefix = lt + la
    for t in tiles + [-1, -17]:   # negative: prefix tiles 0 and 16
        lo = prefix + 64 * t if t >= 0 else 64 * (-t - 1)
        rows = slice(lo, lo + 64)
        raw = [vo.widen(bf16_bits(x[0, rows].cpu().contiguous())) for x in ins]   # identity map
        got = [x[0, rows].float().cpu().double().numpy() for x in out]
        for hh in range(h):
            ref = po.preprocess_rows(raw[0][:, hh], raw[1][:, hh], raw[2][:, hh], raw[3][:, hh],
                                     wq[hh].numpy(), wk[hh].numpy(), 1e-6, cos[rows].numpy(),
                                     sin[rows].numpy(), 96, True)
            _check_qk(got[0][:, hh], ref[0], 96, True, ("q", t, hh))
            _check_qk(got[1][:, hh], ref[1], 96, True, ("k", t, hh))
            assert np.array_equal(got[2][:, hh], ref[2]) and np.array_equal(got[3][:, hh], ref[3])
            if t >= 0:
                for i, name in enumerate(("q", "k", "v")):
                    pooled = views["pooled_" + name][0, hh, t].cpu().double().numpy()
                    mean = got[i][:, hh].mean(axis=0)
                    mabs = np.abs(got[i][:, hh]).mean(axis=0)
                    assert np.all(np.abs(pooled - mean) <= 2.0 ** -18 * mabs + 1e-30), (name, t, hh)
