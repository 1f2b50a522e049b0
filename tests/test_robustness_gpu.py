"""GPU robustness: the forward is capture-safe (CUDA graphs), reads nothing it
has not written or been given, and its output does not depend on stale
workspace or output contents.

* A CUDA-graph capture of vsa_forward replays bit-identically to the eager
  call, and picks up new input values written in place between replays (no
  host reads of device data, no allocation, no synchronisation in the call).
* A workspace filled with 0xFF bytes (NaN in every float, -1 in every index)
  and an output filled with NaN give the same bits as a clean run: every
  buffer is written before it is read.
* Inputs that are views into buffers padded with NaN rows past the last token
  give the same bits as tight buffers: no kernel reads beyond token N.
"""
import pytest
import torch

import block_sparse_video_gb300 as bsv
from block_sparse_video_gb300.synthetic import make_inputs

pytestmark = pytest.mark.gpu


def _bits(x):
    return x.view(torch.int16)


def test_forward_captures_into_a_cuda_graph(cuda_ok):
    shape = (1, 2, 40, 24, 1000)
    q, k, v, g = make_inputs(*shape, 5, device="cuda")
    op = bsv.VSA(*shape, 0.2)
    ref = op(q, k, v, g).clone()
    op.check()

    out = torch.empty_like(ref)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        op(q, k, v, g, out)
    out.fill_(float("nan"))
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    op.check()
    assert torch.equal(_bits(out), _bits(ref))

    # new values in the captured input buffers
    q2, k2, v2, g2 = make_inputs(*shape, 6, device="cuda")
    ref2 = op(q2, k2, v2, g2).clone()
    op.check()
    for dst, src in ((q, q2), (k, k2), (v, v2), (g, g2)):
        dst.copy_(src)
    graph.replay()
    torch.cuda.synchronize()
    op.check()
    assert torch.equal(_bits(out), _bits(ref2))


def test_poisoned_workspace_and_output_do_not_leak(cuda_ok):
    shape = (2, 3, 37, 50, 1000)  # ragged prefix tile and ragged last video tile
    q, k, v, g = make_inputs(*shape, 7, device="cuda")
    op = bsv.VSA(*shape, 0.3)
    ref = op(q, k, v, g).clone()
    op.check()
    op.workspace.fill_(0xFF)
    out = torch.full_like(ref, float("nan"))
    op(q, k, v, g, out)
    op.check()
    assert torch.equal(_bits(out), _bits(ref))


def test_nan_rows_past_the_inputs_are_never_read(cuda_ok):
    shape = (1, 2, 37, 50, 64 * 9 + 11)
    b, h, lt, la, lv = shape
    n = lt + la + lv
    q, k, v, g = make_inputs(*shape, 8, device="cuda")
    op = bsv.VSA(*shape, 0.4)
    ref = op(q, k, v, g).clone()
    op.check()
    padded = []
    for x in (q, k, v, g):
        buf = torch.full((b, n + 192, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        buf[:, :n].copy_(x)
        view = buf[:, :n]
        assert view.is_contiguous()
        padded.append(view)
    out = op(*padded)
    op.check()
    assert torch.equal(_bits(out), _bits(ref))
