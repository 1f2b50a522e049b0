"""GPU tests of the output-row layout ("UniServe: serving FastH3 at its fastest",
section "Fused output combination": the combined rows are written directly
into their positions in the output all-to-all's send buffer).

* Scattering through a row map writes exactly the rows of the packed forward
  (bit for bit: same kernel, other addresses). Rows no token maps to keep
  their contents (NaN-poisoned here).
* A slice of a wider buffer (row stride > H x 128) receives this forward's
  heads and nothing else.
* The serving chain is vsa_preprocess from a capacity-padded projection
  buffer, then vsa_forward_rows back through the same map. It returns every
  row to its sequence position, matches the oracle chain, and replays from a
  CUDA graph.
* An out-of-range entry is skipped and reported.
"""
import numpy as np
import pytest
import torch

import block_sparse_video_gb300 as bsv
from block_sparse_video_gb300.synthetic import (bf16_bits, make_inputs, make_norm_weights, make_projections,
                                                make_rope_tables, make_row_map)
from oracle import preprocess_oracle as po
from oracle import vsa_oracle as vo

pytestmark = pytest.mark.gpu


def _bits(x):
    return x.view(torch.int16)


@pytest.mark.parametrize("subblock", [False, True])
def test_scatter_through_a_row_map_matches_the_packed_forward(cuda_ok, subblock):
    b, h, lt, la, lv = 2, 3, 37, 50, 64 * 6 + 9
    n = lt + la + lv
    q, k, v, g = make_inputs(b, h, lt, la, lv, 40, device="cuda")
    op = bsv.SubBlock(b, h, lt, la, lv, 0.5) if subblock else bsv.VSA(b, h, lt, la, lv, 0.3)
    ref = op(q, k, v, None if subblock else g).clone()
    op.check()
    rows_out = n + 70
    rmap = make_row_map(b, n, rows_out, 41).cuda()
    out = torch.full((b, rows_out, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    op.forward_rows(q, k, v, None if subblock else g, out, rmap)
    op.check()
    for bb in range(b):
        idx = rmap[bb].long()
        assert torch.equal(_bits(out[bb, idx]), _bits(ref[bb]))
        untouched = torch.ones(rows_out, dtype=torch.bool, device="cuda")
        untouched[idx] = False
        assert torch.isnan(out[bb, untouched].float()).all()


def test_head_slice_of_a_wider_buffer(cuda_ok):
    b, h, lt, la, lv = 1, 4, 64, 64, 64 * 5
    n = lt + la + lv
    q, k, v, g = make_inputs(b, h, lt, la, lv, 42, device="cuda")
    op = bsv.VSA(b, h, lt, la, lv, 0.4)
    ref = op(q, k, v, g).clone()
    op.check()
    wide = torch.full((b, n, 3 * h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    view = wide[:, :, h:2 * h]          # this forward's heads, row stride 3 H x 128
    op.forward_rows(q, k, v, g, view)    # no map: token n -> row n
    op.check()
    assert torch.equal(_bits(wide[:, :, h:2 * h]), _bits(ref))
    assert torch.isnan(wide[:, :, :h].float()).all() and torch.isnan(wide[:, :, 2 * h:].float()).all()


def test_bad_output_map_entries_are_skipped_and_reported(cuda_ok):
    b, h, lt, la, lv = 1, 2, 10, 10, 64 * 2
    n = lt + la + lv
    q, k, v, g = make_inputs(b, h, lt, la, lv, 43, device="cuda")
    op = bsv.VSA(b, h, lt, la, lv, 0.5)
    ref = op(q, k, v, g).clone()
    op.check()
    rmap = torch.arange(n, dtype=torch.int32, device="cuda")[None].contiguous()
    rmap[0, 5] = n
    rmap[0, 100] = -1
    out = torch.full((b, n, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    op.forward_rows(q, k, v, g, out, rmap)
    with pytest.raises(bsv.VsaError) as e:
        op.check()
    assert e.value.status == bsv.VSA_ERR_INVALID_ARG
    keep = torch.ones(n, dtype=torch.bool, device="cuda")
    keep[5] = keep[100] = False
    assert torch.equal(_bits(out[0, keep]), _bits(ref[0, keep]))
    assert torch.isnan(out[0, 5].float()).all() and torch.isnan(out[0, 100].float()).all()
    op(q, k, v, g)   # a plain forward clears the report
    op.check()


def test_serving_chain_returns_rows_to_sequence_order_and_replays_from_a_graph(cuda_ok):
    b, h, lt, la, lv = 1, 4, 100, 60, 64 * 12 + 5
    n = lt + la + lv
    rows_in = n + 64                                  # capacity-padded projection buffer
    proj = make_projections(b, rows_in, h, 44, device="cuda")
    ins = [proj[:, :, i] for i in range(4)]
    wq, wk = (w.cuda() for w in make_norm_weights(h, 45))
    cos, sin = (t.cuda() for t in make_rope_tables(lt, la, lv, 96))
    src = make_row_map(b, n, rows_in, 46).cuda()
    op = bsv.VSA(b, h, lt, la, lv, 0.25)
    packed = tuple(torch.empty(op.shape, dtype=torch.bfloat16, device="cuda") for _ in range(4))
    send = torch.full((b, rows_in, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")

    def chain():
        op.preprocess(*ins, wq, wk, cos, sin, 96, True, 1e-6, src, out=packed)
        op.forward_rows(*packed, send, src, preprocessed=True)

    chain()
    op.check()
    first = send.clone()
    # the chain against the oracle chain, two heads: row src[n] holds token n's output
    bits = [bf16_bits(x.cpu().contiguous()) for x in ins]
    pre = po.preprocess(*bits, lt + la, lv, wq.cpu().numpy(), wk.cpu().numpy(), 1e-6, cos.cpu().numpy(),
                        sin.cpu().numpy(), 96, True, src_row=src.cpu().numpy(), heads=[0, 3])
    got = send.float().cpu().double().numpy()
    s = src[0].long().cpu().numpy()
    errs = []
    for hh in (0, 3):
        r = vo.vsa_head(pre["q"][0, :, hh], pre["k"][0, :, hh], pre["v"][0, :, hh], pre["gate"][0, :, hh],
                        lt + la, lv, 0.25)
        errs.append(np.abs(got[0, s, hh] - r["out"]))
    e = np.concatenate(errs)
    assert e.max() <= 2e-2 and e.mean() <= 2e-3, (e.max(), e.mean())
    unmapped = np.setdiff1d(np.arange(rows_in), s)
    assert np.isnan(got[0, unmapped]).all()
    # captured once, replayed: the same bytes
    send.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain()
    send.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    op.check()
    assert torch.equal(_bits(send), _bits(first))
