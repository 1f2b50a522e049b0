"""One rank's head slice of a wider layer, computed in place (GPU, through the
C ABI): "UniServe: serving FastH3 at its fastest", section "The FastH3
workload" (each GPU of the sequence-parallel group attends for its share of
the 56 heads).

A plan of Hr heads reads heads h0 .. h0 + Hr - 1 of [B, N, H, 128] inputs
through vsa_forward_ex's input row stride (H x 128) and writes them into the
same head slice of an [B, N, H, 128] output through output rows. Heads are
independent through the whole forward, so running every rank's slice must give
the full-layer forward's output bit for bit, and one slice must match the
oracle for its heads.
"""
import numpy as np
import pytest
import torch

import block_sparse_video_gb300 as bsv
from block_sparse_video_gb300.sharding import head_ranges
from block_sparse_video_gb300.synthetic import bf16_bits, make_inputs
from tests.vsa_parity import assert_errors, compare_head, to_f64

pytestmark = pytest.mark.gpu


def _bits(x):
    return x.view(torch.int16)


@pytest.mark.parametrize("subblock", [False, True])
@pytest.mark.parametrize("world", [2, 4])
def test_rank_slices_rebuild_the_full_layer(cuda_ok, subblock, world):
    b, h, lt, la, lv = 2, 6, 70, 33, 64 * 9 + 17
    q, k, v, g = make_inputs(b, h, lt, la, lv, 160 + world, device="cuda")
    gate = None if subblock else g

    def plan(heads):
        return bsv.SubBlock(b, heads, lt, la, lv, 0.6) if subblock else bsv.VSA(b, heads, lt, la, lv, 0.25)

    full_op = plan(h)
    full = full_op.forward_ex(q, k, v, gate)
    full_op.check()
    out = torch.full_like(q, float("nan"))
    for h0, n in head_ranges(h, world):
        op = plan(n)
        s = slice(h0, h0 + n)
        op.forward_ex(q[:, :, s], k[:, :, s], v[:, :, s], None if subblock else g[:, :, s], out=out[:, :, s])
        op.check()
    assert torch.equal(_bits(out), _bits(full))


def test_one_slice_matches_the_oracle(cuda_ok):
    b, h, lt, la, lv = 1, 7, 64, 64, 64 * 14 + 3
    h0, n = head_ranges(h, 3)[1]          # heads 3 .. 4
    q, k, v, g = make_inputs(b, h, lt, la, lv, 170, device="cuda")
    op = bsv.VSA(b, n, lt, la, lv, 0.2)
    s = slice(h0, h0 + n)
    out = torch.full_like(q, float("nan"))
    op.forward_ex(q[:, :, s], k[:, :, s], v[:, :, s], g[:, :, s], out=out[:, :, s])
    op.check()
    assert torch.isnan(out[:, :, :h0].float()).all() and torch.isnan(out[:, :, h0 + n:].float()).all()
    views = {name: t.cpu() for name, t in op.debug_views().items()}
    sl_bits = [bf16_bits(x[:, :, s].contiguous().cpu()) for x in (q, k, v, g)]
    o = to_f64(out[:, :, s].contiguous())
    stats = [compare_head(*sl_bits, views, o, 0, hh, lt + la, lv, 0.2) for hh in range(n)]
    assert_errors(stats, "head slice 3..4 of 7")


def test_slice_with_device_lengths(cuda_ok):
    """A head slice of a capacity-padded buffer, lengths read on the device."""
    b, h, cap = 1, 4, (100, 40, 64 * 8 + 9)
    req = (60, 40, 64 * 5 + 1)
    n_cap, n = sum(cap), sum(req)
    q, k, v, g = make_inputs(b, h, *req, 175, device="cuda")
    bufs = [torch.full((b, n_cap, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    for dst, src in zip(bufs, (q, k, v, g)):
        dst[:, :n].copy_(src)
    ref_op = bsv.VSA(b, h, *req, 0.25)
    ref = ref_op(q, k, v, g)
    ref_op.check()
    lengths = torch.tensor(list(req), dtype=torch.int64, device="cuda")
    out = torch.full((b, n_cap, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    for h0, cnt in head_ranges(h, 2):
        op = bsv.VSA(b, cnt, *cap, 0.25)
        s = slice(h0, h0 + cnt)
        op.forward_ex(*(x[:, :, s] for x in bufs), out=out[:, :, s], lengths=lengths)
        op.check()
    assert torch.equal(_bits(out[:, :n]), _bits(ref))
    assert torch.isnan(out[:, n:].float()).all()


def test_mixed_row_strides_are_rejected(cuda_ok):
    b, h, lt, la, lv = 1, 4, 64, 0, 256
    q, k, v, g = make_inputs(b, h, lt, la, lv, 180, device="cuda")
    op = bsv.VSA(b, 2, lt, la, lv, 0.25)
    packed = q[:, :, :2].contiguous()
    with pytest.raises(ValueError):
        op.forward_ex(packed, k[:, :, :2], v[:, :, :2], g[:, :, :2])
