"""The capacity-padded forward (device-side lengths) against the CPU oracle,
with NaN in every padding row ("UniServe: serving FastH3 at its fastest",
sections "Architecture": one workspace for the largest shape and device-side
index tensors per shape bucket; and "Fused attention preprocessing": padding
is handled inside the kernel, so it never becomes an input to later steps).

Each request sits at the top of [B, N_cap, H, 128] buffers whose rows N ..
N_cap - 1 hold NaN. The request's output rows are compared with the oracle
run on the request's exact tensors (every batch, head and row), intermediates
included; output rows past N must stay untouched. Requests cover a ragged
prefix and a ragged last video tile, no prefix, exactly the capacity, a single
video token, and a ragged prefix tile whose 64-row load reaches past the
request's last token. The serving step (preprocessing from a capacity-padded
projection buffer, the forward, rows written back to their sequence positions)
runs against the preprocessing and VSA oracles the same way.
"""
import numpy as np
import pytest
import torch

import block_sparse_video_gb300 as bsv
from block_sparse_video_gb300.synthetic import (bf16_bits, make_inputs, make_norm_weights, make_projections,
                                                make_rope_tables, make_row_map)
from oracle import preprocess_oracle as po
from oracle import subblock_oracle as so
from oracle import vsa_oracle as vo
from tests.test_subblock_gpu import _check_selection as check_subblock_selection
from tests.vsa_parity import assert_errors, compare_head, to_f64

pytestmark = pytest.mark.gpu

CAP = (2, 3, 130, 70, 64 * 12 + 30)   # batch, heads, text, audio, video
KEEP = 0.25
SPARSITY = 0.6
REQUESTS = [
    (100, 50, 64 * 9 + 5),     # ragged prefix and ragged last tile
    (0, 0, 64 * 5),            # no prefix
    (130, 70, 64 * 12 + 30),   # exactly the capacity
    (64, 64, 1),               # one video token
    (100, 0, 5),               # the ragged prefix tile's rows 105 .. 127 are padding
    (7, 0, 64 * 12 + 30),      # text only, full video
]


def _nan_buffers(shape, n):
    return [torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(n)]


def _sliced_views(views, t, k):
    """The request's part of a capacity plan's views: the first t tiles of each
    [T_cap] block and the first k selections of each row."""
    out = {name: x[:, :, :t] for name, x in views.items() if x is not None and name != "tile_index"}
    out["tile_index"] = views["tile_index"][:, :, :t, :k]
    return out


@pytest.mark.parametrize("req", REQUESTS, ids=[f"{a}+{b}+{c}" for a, b, c in REQUESTS])
def test_capacity_forward_matches_oracle_with_nan_padding(cuda_ok, req):
    b, h, clt, cla, clv = CAP
    lt, la, lv = req
    n = lt + la + lv
    cap = bsv.VSA(b, h, clt, cla, clv, KEEP)
    bufs = _nan_buffers(cap.shape, 4)
    q, k, v, g = make_inputs(b, h, lt, la, lv, 120 + n, device="cuda")
    for dst, src in zip(bufs, (q, k, v, g)):
        dst[:, :n].copy_(src)
    lengths = torch.tensor([lt, la, lv], dtype=torch.int64, device="cuda")
    out = torch.full(cap.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    cap.forward_lengths(lengths, *bufs, out)
    cap.check()
    assert torch.isfinite(out[:, :n].float()).all()
    assert torch.isnan(out[:, n:].float()).all()
    t = vo.video_tile_count(lv)
    kk = vo.keep_count(t, KEEP)
    views = _sliced_views({name: x.cpu() for name, x in cap.debug_views().items()}, t, kk)
    bits = [bf16_bits(x.cpu()) for x in (q, k, v, g)]
    o = to_f64(out[:, :n])
    stats = [compare_head(*bits, views, o, bb, hh, lt + la, lv, KEEP) for bb in range(b) for hh in range(h)]
    assert_errors(stats, f"capacity request {req}")


@pytest.mark.parametrize("req", REQUESTS, ids=[f"{a}+{b}+{c}" for a, b, c in REQUESTS])
def test_capacity_subblock_forward_matches_oracle_with_nan_padding(cuda_ok, req):
    b, h, clt, cla, clv = CAP
    lt, la, lv = req
    n = lt + la + lv
    cap = bsv.SubBlock(b, h, clt, cla, clv, SPARSITY)
    bufs = _nan_buffers(cap.shape, 3)
    q, k, v, _ = make_inputs(b, h, lt, la, lv, 140 + n, device="cuda")
    for dst, src in zip(bufs, (q, k, v)):
        dst[:, :n].copy_(src)
    lengths = torch.tensor([lt, la, lv], dtype=torch.int64, device="cuda")
    out = torch.full(cap.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    cap.forward_lengths(lengths, *bufs, None, out)
    cap.check()
    assert torch.isfinite(out[:, :n].float()).all()
    assert torch.isnan(out[:, n:].float()).all()
    t = vo.video_tile_count(lv)
    kk = so.keep_count(t, SPARSITY)
    views = {name: x.cpu() for name, x in cap.debug_views().items() if x is not None}
    idx = views["tile_index"][:, :, :t, :kk].numpy()
    bits = [bf16_bits(x.cpu()) for x in (q, k, v)]
    o = to_f64(out[:, :n])
    stats = []
    for bb in range(b):
        for hh in range(h):
            args = (bits[0][bb, :, hh], bits[1][bb, :, hh], bits[2][bb, :, hh])
            r = so.subblock_head(*args, lt + la, lv, SPARSITY, video_tiles=[], prefix_rows=[])
            np.testing.assert_allclose(views["sub_q"][bb, hh, :4 * t].numpy(), r["sub_q"], rtol=2e-6, atol=2e-6)
            overrides = check_subblock_selection(idx[bb, hh], r["index"], r["scores"], r["k"])
            r = so.subblock_head(*args, lt + la, lv, SPARSITY, index_override=overrides)
            err = np.abs(o[bb, :, hh] - r["out"])
            stats.append(dict(max_abs=float(err.max()), sum_abs=float(err.sum()), count=int(err.size)))
    assert_errors(stats, f"SubBlock capacity request {req}")


def test_serving_step_in_capacity_matches_oracle_with_nan_padding(cuda_ok):
    """vsa_preprocess from a capacity-padded projection buffer (NaN in every row
    no token maps to), then vsa_forward_ex with device lengths over packed
    buffers whose padding rows are NaN, writing rows back through the map;
    compared with the preprocessing oracle followed by the VSA oracle."""
    b, h = 1, 3
    cap_lt, cap_la, cap_lv = 100, 60, 64 * 12 + 5
    cap = bsv.VSA(b, h, cap_lt, cap_la, cap_lv, KEEP)
    n_cap = cap.seq
    rows_in = n_cap + 64
    wq, wk = (w.cuda() for w in make_norm_weights(h, 150))
    for i, (lt, la, lv) in enumerate([(100, 60, 64 * 12 + 5), (37, 0, 64 * 7 + 1), (90, 0, 9)]):
        n = lt + la + lv
        src = make_row_map(b, n, rows_in, 151 + i).cuda()
        proj = make_projections(b, rows_in, h, 155 + i, device="cuda")
        unmapped = torch.ones(rows_in, dtype=torch.bool, device="cuda")
        unmapped[src[0].long()] = False
        proj[:, unmapped] = float("nan")
        ins = [proj[:, :, j] for j in range(4)]
        c, s_ = make_rope_tables(lt, la, lv, 96)
        cos = torch.full((n_cap, 48), float("nan"), dtype=torch.float32, device="cuda")
        sin = torch.full((n_cap, 48), float("nan"), dtype=torch.float32, device="cuda")
        cos[:n].copy_(c)
        sin[:n].copy_(s_)
        src_cap = torch.zeros((b, n_cap), dtype=torch.int32, device="cuda")
        src_cap[:, :n].copy_(src)
        packed = tuple(_nan_buffers(cap.shape, 4))
        send = torch.full((b, rows_in, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        lengths = torch.tensor([lt, la, lv], dtype=torch.int64, device="cuda")
        cap.preprocess(*ins, wq, wk, cos, sin, 96, True, 1e-6, src_cap, out=packed, lengths=lengths)
        cap.forward_ex(*packed, out=send, out_row_map=src_cap, lengths=lengths, preprocessed=True)
        cap.check()
        assert torch.isnan(packed[0][:, n:].float()).all()  # padding stays padding
        bits = [bf16_bits(x.cpu().contiguous()) for x in ins]
        pre = po.preprocess(*bits, lt + la, lv, wq.cpu().numpy(), wk.cpu().numpy(), 1e-6, c.numpy(), s_.numpy(),
                            96, True, src_row=src.cpu().numpy())
        got = send.float().cpu().double().numpy()
        rows = src[0].long().cpu().numpy()
        stats = []
        for hh in range(h):
            r = vo.vsa_head(pre["q"][0, :, hh], pre["k"][0, :, hh], pre["v"][0, :, hh], pre["gate"][0, :, hh],
                            lt + la, lv, KEEP)
            err = np.abs(got[0, rows, hh] - r["out"])
            stats.append(dict(max_abs=float(err.max()), sum_abs=float(err.sum()), count=int(err.size)))
        assert_errors(stats, f"serving step {lt}+{la}+{lv}")
        assert np.isnan(got[0, np.setdiff1d(np.arange(rows_in), rows)]).all()
