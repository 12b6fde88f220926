"""Failure detection on the GPU without a GPU fault.

Every mbarrier wait in the tensor-core kernels is bounded. The test starves one
wait: the forward's producer arms a pipeline stage but never issues its loads,
a flag nothing sets (armed for this host thread by flce_test_fault). It checks
three things:
- the kernel gives up after the (shortened) limit and reports FLCE_ERR_TIMEOUT
  through the workspace status word;
- it frees its tensor memory and returns, with no trap, no fault and no hang;
- the same process then runs a correct forward on the same GPU.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_cross_entropy_tiled_gb300 import _lib
from linear_cross_entropy_tiled_gb300.functional import flce_forward
from linear_cross_entropy_tiled_gb300.workloads import small_case

from flce_check import assert_loss_close, to_device

pytestmark = pytest.mark.gpu


def test_starved_wait_reports_timeout_and_the_context_survives():
    d = small_case(600, 256, 3000, seed=17, dtype="bf16", bias=True, ignore_frac=0.1)
    h, w, b, t = to_device(d, "bf16")
    p = _lib.make_params(N=600, H=256, V=3000, dtype=_lib.FLCE_BF16, has_bias=True,
                         reduction="mean")
    stream = torch.cuda.current_stream().cuda_stream
    _lib.test_fault(1, 100)
    try:
        loss, lse, nc, ent, ws = flce_forward(p, h, w, t, b, return_metrics=True)
    finally:
        _lib.test_fault(-1, 0)
    assert _lib.check_status(ws.data_ptr(), stream) == 7          # FLCE_ERR_TIMEOUT
    # nothing of the aborted forward looks like a result
    assert np.isnan(loss.item()) and np.isnan(lse.cpu().numpy()).all()
    assert nc.item() == -1 and np.isnan(ent.item())
    loss, _, _, _, ws = flce_forward(p, h, w, t, b)
    assert _lib.check_status(ws.data_ptr(), stream) == 0
    ref = oracle.forward(d["hidden"], d["weight"], d["targets"], bias=d["bias"], reduction="mean")
    assert_loss_close(loss.cpu().numpy(), ref["loss"], "bf16")
