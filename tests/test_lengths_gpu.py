"""GPU tests of the capacity-padded forward with device-side lengths
("UniServe: serving FastH3 at its fastest", section "Architecture": one
workspace for the largest shape, CUDA graphs captured once per shape bucket
and addressing each request through device-side tensors).

* A plan's shape is the capacity. Each request's rows sit at the top of
  [B, N_cap, H, 128] buffers whose padding rows hold finite garbage. Rows
  0 .. N - 1 of the output must equal, bit for bit, the forward of an
  exact-shape plan on the exact tensors (same items, same key sets, same
  order). Padding rows of the output stay untouched.
* One captured graph replays every request of the bucket. Lengths and inputs
  are rewritten in place between replays.
* Lengths outside the capacity compute nothing and are reported.
"""
import pytest
import torch

import block_sparse_video_gb300 as bsv
from block_sparse_video_gb300.synthetic import make_inputs

pytestmark = pytest.mark.gpu

CAP = (2, 3, 130, 70, 64 * 12 + 30)   # batch, heads, text, audio, video
KEEP = 0.25
SPARSITY = 0.6
REQUESTS = [
    (100, 50, 64 * 9 + 5),     # ragged prefix and ragged last tile
    (0, 0, 64 * 5),            # no prefix
    (130, 70, 64 * 12 + 30),   # exactly the capacity
    (64, 64, 1),               # one video token
    (7, 0, 64 * 12 + 30),      # text only, full video
]


def _bits(x):
    return x.view(torch.int16)


def _capacity_buffers(b, h, n_cap, seed):
    """Four [B, N_cap, H, 128] bf16 tensors of finite garbage."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    return [torch.randn((b, n_cap, h, 128), generator=gen, device="cuda").to(torch.bfloat16) for _ in range(4)]


def _exact(b, h, lt, la, lv, seed):
    q, k, v, g = make_inputs(b, h, lt, la, lv, seed, device="cuda")
    op = bsv.VSA(b, h, lt, la, lv, KEEP)
    out = op(q, k, v, g).clone()
    op.check()
    return (q, k, v, g), out


def test_each_request_matches_an_exact_shape_plan(cuda_ok):
    b, h, clt, cla, clv = CAP
    cap = bsv.VSA(b, h, clt, cla, clv, KEEP)
    n_cap = cap.seq
    bufs = _capacity_buffers(b, h, n_cap, 50)
    lengths = torch.empty(3, dtype=torch.int64, device="cuda")
    for i, (lt, la, lv) in enumerate(REQUESTS):
        n = lt + la + lv
        ins, ref = _exact(b, h, lt, la, lv, 60 + i)
        for dst, src in zip(bufs, ins):
            dst[:, :n].copy_(src)
        lengths.copy_(torch.tensor([lt, la, lv]))
        out = torch.full((b, n_cap, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        cap.forward_lengths(lengths, *bufs, out)
        cap.check()
        assert torch.equal(_bits(out[:, :n]), _bits(ref)), (lt, la, lv)
        assert torch.isnan(out[:, n:].float()).all(), (lt, la, lv)


def test_one_captured_graph_serves_every_request(cuda_ok):
    b, h, clt, cla, clv = CAP
    cap = bsv.VSA(b, h, clt, cla, clv, KEEP)
    n_cap = cap.seq
    bufs = _capacity_buffers(b, h, n_cap, 51)
    out = torch.full((b, n_cap, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lengths = torch.tensor(list(REQUESTS[0]), dtype=torch.int64, device="cuda")
    cap.forward_lengths(lengths, *bufs, out)  # warm-up outside the capture
    cap.check()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap.forward_lengths(lengths, *bufs, out)
    for i, (lt, la, lv) in enumerate(REQUESTS[::-1]):
        n = lt + la + lv
        ins, ref = _exact(b, h, lt, la, lv, 70 + i)
        for dst, src in zip(bufs, ins):
            dst[:, :n].copy_(src)
        lengths.copy_(torch.tensor([lt, la, lv]))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        cap.check()
        assert torch.equal(_bits(out[:, :n]), _bits(ref)), (lt, la, lv)
        assert torch.isnan(out[:, n:].float()).all()


@pytest.mark.parametrize("bad", [(131, 70, 64), (0, 0, 0), (0, 0, 64 * 12 + 31), (-1, 5, 64), (100, 101, 64)])
def test_lengths_outside_the_capacity_are_reported(cuda_ok, bad):
    b, h, clt, cla, clv = CAP
    cap = bsv.VSA(b, h, clt, cla, clv, KEEP)
    bufs = _capacity_buffers(b, h, cap.seq, 52)
    out = torch.full((b, cap.seq, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lengths = torch.tensor(list(bad), dtype=torch.int64, device="cuda")
    cap.forward_lengths(lengths, *bufs, out)
    with pytest.raises(bsv.VsaError) as e:
        cap.check()
    assert e.value.status == bsv.VSA_ERR_INVALID_ARG
    assert torch.isnan(out.float()).all()
    lengths.copy_(torch.tensor(list(REQUESTS[0])))   # the next valid request clears the report
    cap.forward_lengths(lengths, *bufs, out)
    cap.check()


def test_page_requests_in_the_10s_capacity_buffer(cuda_ok):
    """The page's 10 s request (1,000 text + 810 audio + 72,576 video tokens) and
    a 5 s-like request in one 78,080-row capacity plan (56 heads), replayed from
    one graph; both equal exact-shape plans bit for bit."""
    b, h = 1, 56
    cap = bsv.VSA(b, h, 1024, 1024, 76032, 0.2)     # 78,080 rows
    assert cap.seq == 78080
    bufs = _capacity_buffers(b, h, cap.seq, 53)
    out = torch.empty((b, cap.seq, h, 128), dtype=torch.bfloat16, device="cuda")
    lengths = torch.tensor([1000, 810, 72576], dtype=torch.int64, device="cuda")
    cap.forward_lengths(lengths, *bufs, out)
    cap.check()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap.forward_lengths(lengths, *bufs, out)
    for i, (lt, la, lv) in enumerate([(1000, 810, 72576), (1024, 1024, 36288)]):
        n = lt + la + lv
        q, k, v, g = make_inputs(b, h, lt, la, lv, 80 + i, device="cuda")
        for dst, src in zip(bufs, (q, k, v, g)):
            dst[:, :n].copy_(src)
        lengths.copy_(torch.tensor([lt, la, lv]))
        graph.replay()
        torch.cuda.synchronize()
        cap.check()
        op = bsv.VSA(b, h, lt, la, lv, 0.2)
        ref = op(q, k, v, g)
        op.check()
        assert torch.equal(_bits(out[:, :n]), _bits(ref)), (lt, la, lv)
        del q, k, v, g, ref, op
        torch.cuda.empty_cache()


@pytest.mark.parametrize("subblock", [False, True])
def test_serving_step_in_one_graph(cuda_ok, subblock):
    """The serving step of one layer replayed from a single captured graph for
    requests of different lengths (device-side lengths throughout):
      1. vsa_preprocess packs and normalises the request from a capacity-padded
         projection buffer through its row map;
      2. vsa_forward_ex attends over the packed tensors (VSA selection, or the
         SubBlock router with no gate);
      3. it writes each combined row back to its sequence position, the output
         all-to-all's send layout.
    Each replay equals the same chain on an exact-shape plan, bit for bit."""
    from block_sparse_video_gb300.synthetic import make_norm_weights, make_projections, make_rope_tables, make_row_map
    b, h = 1, 4
    cap_lt, cap_la, cap_lv = 100, 60, 64 * 12 + 5

    def plan(lt, la, lv):
        return bsv.SubBlock(b, h, lt, la, lv, SPARSITY) if subblock else bsv.VSA(b, h, lt, la, lv, KEEP)

    cap = plan(cap_lt, cap_la, cap_lv)
    n_cap = cap.seq
    rows_in = n_cap + 64
    proj = torch.zeros((b, rows_in, 4, h, 128), dtype=torch.bfloat16, device="cuda")
    ins = [proj[:, :, i] for i in range(4)]
    wq, wk = (w.cuda() for w in make_norm_weights(h, 90))
    cos = torch.zeros((n_cap, 48), dtype=torch.float32, device="cuda")
    sin = torch.zeros((n_cap, 48), dtype=torch.float32, device="cuda")
    src = torch.zeros((b, n_cap), dtype=torch.int32, device="cuda")
    packed = tuple(torch.zeros(cap.shape, dtype=torch.bfloat16, device="cuda") for _ in range(4))
    send = torch.full((b, rows_in, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lengths = torch.tensor([cap_lt, cap_la, cap_lv], dtype=torch.int64, device="cuda")

    def step():
        cap.preprocess(*ins, wq, wk, cos, sin, 96, True, 1e-6, src, out=packed, lengths=lengths)
        cap.forward_ex(*packed[:3], None if subblock else packed[3], out=send, out_row_map=src, lengths=lengths,
                       preprocessed=True)

    step()
    cap.check()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for i, (lt, la, lv) in enumerate([(100, 60, 64 * 12 + 5), (37, 0, 64 * 7 + 1), (64, 50, 300)]):
        n = lt + la + lv
        proj.copy_(make_projections(b, rows_in, h, 91 + i, device="cuda"))
        c, s_ = make_rope_tables(lt, la, lv, 96)
        cos[:n].copy_(c)
        sin[:n].copy_(s_)
        src[:, :n].copy_(make_row_map(b, n, rows_in, 95 + i))
        lengths.copy_(torch.tensor([lt, la, lv]))
        send.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        cap.check()
        # the exact-shape chain on the same data
        ex = plan(lt, la, lv)
        ex_send = torch.full_like(send, float("nan"))
        ex_src = src[:, :n].contiguous()
        pk = ex.preprocess(*ins, wq, wk, cos[:n].contiguous(), sin[:n].contiguous(), 96, True, 1e-6, ex_src)
        ex.forward_rows(*pk[:3], None if subblock else pk[3], ex_send, ex_src, preprocessed=True)
        ex.check()
        assert torch.equal(_bits(send), _bits(ex_send)), (lt, la, lv)
        assert torch.isnan(send.float()).sum() == (rows_in - n) * h * 128 * b



def _exact_subblock(b, h, lt, la, lv, seed):
    q, k, v, _ = make_inputs(b, h, lt, la, lv, seed, device="cuda")
    op = bsv.SubBlock(b, h, lt, la, lv, SPARSITY)
    out = op(q, k, v).clone()
    op.check()
    return (q, k, v), out, op.debug_views()["tile_index"].clone()


def test_subblock_requests_match_exact_shape_plans(cuda_ok):
    """SubBlock routing in a capacity plan: the sub-block pool and the router
    read the device lengths too (k from the request's T: T - floor(s T) rounded
    up to 8, capped at T). Each request equals an exact-shape SubBlock plan bit
    for bit, selections included; padding rows stay untouched."""
    b, h, clt, cla, clv = CAP
    cap = bsv.SubBlock(b, h, clt, cla, clv, SPARSITY)
    n_cap = cap.seq
    bufs = _capacity_buffers(b, h, n_cap, 54)[:3]
    lengths = torch.empty(3, dtype=torch.int64, device="cuda")
    for i, (lt, la, lv) in enumerate(REQUESTS):
        n = lt + la + lv
        ins, ref, ref_idx = _exact_subblock(b, h, lt, la, lv, 90 + i)
        for dst, src in zip(bufs, ins):
            dst[:, :n].copy_(src)
        lengths.copy_(torch.tensor([lt, la, lv]))
        out = torch.full((b, n_cap, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        cap.forward_lengths(lengths, *bufs, None, out)
        cap.check()
        t, kk = ref_idx.shape[2], ref_idx.shape[3]
        assert torch.equal(cap.debug_views()["tile_index"][:, :, :t, :kk], ref_idx), (lt, la, lv)
        assert torch.equal(_bits(out[:, :n]), _bits(ref)), (lt, la, lv)
        assert torch.isnan(out[:, n:].float()).all(), (lt, la, lv)


def test_one_captured_graph_serves_every_subblock_request(cuda_ok):
    b, h, clt, cla, clv = CAP
    cap = bsv.SubBlock(b, h, clt, cla, clv, SPARSITY)
    n_cap = cap.seq
    bufs = _capacity_buffers(b, h, n_cap, 55)[:3]
    out = torch.full((b, n_cap, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lengths = torch.tensor(list(REQUESTS[0]), dtype=torch.int64, device="cuda")
    cap.forward_lengths(lengths, *bufs, None, out)  # warm-up outside the capture
    cap.check()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap.forward_lengths(lengths, *bufs, None, out)
    for i, (lt, la, lv) in enumerate(REQUESTS[::-1]):
        n = lt + la + lv
        ins, ref, _ = _exact_subblock(b, h, lt, la, lv, 100 + i)
        for dst, src in zip(bufs, ins):
            dst[:, :n].copy_(src)
        lengths.copy_(torch.tensor([lt, la, lv]))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        cap.check()
        assert torch.equal(_bits(out[:, :n]), _bits(ref)), (lt, la, lv)
        assert torch.isnan(out[:, n:].float()).all()


@pytest.mark.parametrize("bad", [(131, 70, 64), (0, 0, 0), (0, 0, 64 * 12 + 31)])
def test_subblock_lengths_outside_the_capacity_are_reported(cuda_ok, bad):
    b, h, clt, cla, clv = CAP
    cap = bsv.SubBlock(b, h, clt, cla, clv, SPARSITY)
    bufs = _capacity_buffers(b, h, cap.seq, 56)[:3]
    out = torch.full((b, cap.seq, h, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lengths = torch.tensor(list(bad), dtype=torch.int64, device="cuda")
    cap.forward_lengths(lengths, *bufs, None, out)
    with pytest.raises(bsv.VsaError) as e:
        cap.check()
    assert e.value.status == bsv.VSA_ERR_INVALID_ARG
    assert torch.isnan(out.float()).all()
    lengths.copy_(torch.tensor(list(REQUESTS[0])))   # the next valid request clears the report
    cap.forward_lengths(lengths, *bufs, None, out)
    cap.check()
