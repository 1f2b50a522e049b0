"""The forward entry point that allocates nothing (vsa_forward_static_workspace).

Some callers of this library cannot allocate device memory: a serving engine
that budgets all device memory at start-up, a plugin interface that hands a
kernel only its input and output buffers, or a latency-critical path that
must not call cudaMalloc. For them the library keeps its scratch in a
fixed-size device array of its own. These tests call that entry point through
the C ABI and check it against the regular forward (which takes a caller
workspace), twice in a row, since the shared array keeps the previous call's
contents. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import block_sparse_video_gb300 as bsv
from block_sparse_video_gb300.synthetic import make_inputs

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


@pytest.mark.parametrize("shape", [
    (1, 14, 1024, 512, 8192, 0.2, 1),   # medium workload
    (1, 14, 1024, 1024, 36288, 0.2, 2), # one GPU's head share of a 5 s request
    (2, 3, 37, 50, 1000, 0.3, 5),       # ragged prefix and last tile, batch 2
])
def test_static_workspace_forward_matches_regular_forward(cuda_ok, shape):
    b, h, lt, la, lv, keep, seed = shape
    q, k, v, g = make_inputs(b, h, lt, la, lv, seed, device="cuda")
    op = bsv.VSA(b, h, lt, la, lv, keep)
    assert op.workspace_bytes <= bsv.STATIC_WORKSPACE_BYTES
    ref = op(q, k, v, g)
    op.check()
    ref = ref.float()
    for _ in range(2):  # the second call sees the first call's leftovers in the shared array
        out = torch.full_like(q, float("nan"))
        bsv.vsa_forward_static_workspace(op.plan, q, k, v, g, out)
        torch.cuda.synchronize()
        err = (out.float() - ref).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS


def test_static_workspace_rejects_plans_that_do_not_fit(cuda_ok):
    plan = bsv.vsa_plan_create(1, 56, 1024, 1024, 72576, 0.2)  # the 10 s shape needs ~334 MB
    try:
        assert bsv.vsa_plan_info(plan)[2] > bsv.STATIC_WORKSPACE_BYTES
        x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
        p = ctypes.c_void_p(x.data_ptr())
        status = bsv.load_library().vsa_forward_static_workspace(plan, p, p, p, p, p, None)
        assert status == bsv.VSA_ERR_UNSUPPORTED
        with pytest.raises(bsv.VsaError, match="exceeds"):
            bsv.vsa_forward_static_workspace(plan, x, x, x, x, x)
    finally:
        bsv.vsa_plan_destroy(plan)


def test_static_workspace_reports_device_errors(cuda_ok):
    """The library-owned array keeps the forward's error words; the check that
    goes with the entry point reads them (a bounded wait that ran out is planted
    by the diagnostic kernel, no GPU fault), and the next forward starts clean."""
    b, h, lt, la, lv, keep = 1, 2, 64, 64, 1024, 0.2
    q, k, v, g = make_inputs(b, h, lt, la, lv, 0, device="cuda")
    op = bsv.VSA(b, h, lt, la, lv, keep)
    ref = op(q, k, v, g).clone()
    op.check()
    out = torch.empty_like(q)
    bsv.vsa_forward_static_workspace(op.plan, q, k, v, g, out)
    bsv.vsa_check_static_workspace(op.plan)
    bsv.vsa_diag_wait_timeout_static(op.plan, n_ctas=4)
    with pytest.raises(bsv.VsaError) as exc:
        bsv.vsa_check_static_workspace(op.plan)
    assert exc.value.status == bsv.VSA_ERR_DEVICE_TIMEOUT
    out = torch.full_like(q, float("nan"))
    bsv.vsa_forward_static_workspace(op.plan, q, k, v, g, out)
    bsv.vsa_check_static_workspace(op.plan)
    err = (out.float() - ref.float()).abs()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
