"""Failure detection on the GPU without a fault: bounded waits run out, the
kernel records VSA_ERR_DEVICE_TIMEOUT, other CTAs stop on the abort flag, and
the context stays usable for the next forward."""
import time

import pytest
import torch

import block_sparse_video_gb300 as bsv
from block_sparse_video_gb300.synthetic import make_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_ok):
    q, k, v, g = make_inputs(1, 2, 64, 64, 1024, 0, device="cuda")
    op = bsv.VSA(1, 2, 64, 64, 1024, 0.2)
    ref = op(q, k, v, g).clone()
    op.check()
    t0 = time.time()
    bsv.vsa_diag_wait_timeout(op.plan, op.workspace, n_ctas=600)
    with pytest.raises(bsv.VsaError) as exc:
        op.check()
    elapsed = time.time() - t0
    assert exc.value.status == bsv.VSA_ERR_DEVICE_TIMEOUT
    assert elapsed < 10.0, f"600 waiting CTAs took {elapsed:.1f} s: the abort flag did not stop them"
    out = op(q, k, v, g)  # the next forward clears the error words and runs normally
    op.check()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
