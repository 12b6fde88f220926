"""flce_forward_noalloc: the forward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: frameworks that forbid allocation once
their memory plan is fixed, runtimes that hand out memory only from a fixed
arena, plain C hosts holding only their tensors' pointers. For them the
library keeps the forward scratch in one fixed device array of its own
instead of a caller workspace. These tests call that entry point through the
C ABI:
- twice in a row, on different inputs, so stale scratch would show. Each
  result must equal, bit for bit, the workspace-taking flce_forward on the
  same inputs and stream (the kernels are the same), and match the fp64
  oracle within the parity tolerances of the other GPU tests;
- with a starved pipeline stage (flce_test_fault, a bounded wait that runs
  out; nothing faults). The array then still holds the previous call's
  partial states, and the outputs must be NaN (num_correct -1), not a
  plausible stale loss. The next call must be correct again;
- with a size whose scratch exceeds the fixed maximum, which is refused
  before any kernel launches.

The file name sorts last, so a run that stops at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_cross_entropy_tiled_gb300 import _lib
from linear_cross_entropy_tiled_gb300.functional import flce_forward
from linear_cross_entropy_tiled_gb300.workloads import small_case

from flce_check import assert_entropy_close, assert_loss_close, assert_lse_close, to_device

pytestmark = pytest.mark.gpu

SCRATCH_MAX = 48 << 20   # the fixed array size stated in include/flce.h


def noalloc_forward(p, h, w, b, t):
    dev = h.device
    nloss = p.N if p.reduction == _lib.FLCE_NONE else 1
    loss = torch.empty(nloss, dtype=torch.float32, device=dev)
    lse = torch.empty(p.N, dtype=torch.float32, device=dev)
    nc = torch.empty(1, dtype=torch.int64, device=dev)
    ent = torch.empty(1, dtype=torch.float32, device=dev)
    rc = _lib.forward_noalloc_raw(p, h.data_ptr(), w.data_ptr(), 0 if b is None else b.data_ptr(),
                                  t.data_ptr(), loss.data_ptr(), lse.data_ptr(), nc.data_ptr(),
                                  ent.data_ptr(), torch.cuda.current_stream(dev).cuda_stream)
    _lib.check(rc, "flce_forward_noalloc")
    torch.cuda.synchronize(dev)
    return loss.cpu().numpy(), lse.cpu().numpy(), int(nc.item()), float(ent.item())


CASES = [
    dict(N=700, H=264, V=1300, seed=31, bias=True, kw=dict(reduction="mean", softcap=20.0,
                                                           z_loss_multiplier=1e-4)),
    dict(N=333, H=136, V=2053, seed=32, bias=False, kw=dict(reduction="none", logit_scale=0.7)),
]


def setup(c):
    d = small_case(c["N"], c["H"], c["V"], seed=c["seed"], dtype="bf16", bias=c["bias"],
                   ignore_frac=0.1)
    h, w, b, t = to_device(d, "bf16")
    p = _lib.make_params(N=c["N"], H=c["H"], V=c["V"], dtype=_lib.FLCE_BF16,
                         has_bias=c["bias"], **c["kw"])
    assert _lib.workspace_bytes(p, _lib.FLCE_PASS_FORWARD) <= SCRATCH_MAX
    return d, p, (h, w, b, t)


def check_against_workspace_forward_and_oracle(c, d, p, dev, got):
    h, w, b, t = dev
    loss, lse, nc, ent = got
    rl, rlse, rnc, rent, _ = flce_forward(p, h, w, t, b, return_metrics=True)
    torch.cuda.synchronize()
    # the same kernels on the same inputs: identical bits
    np.testing.assert_array_equal(loss, rl.cpu().numpy())
    np.testing.assert_array_equal(lse, rlse.cpu().numpy())
    assert nc == int(rnc.item())
    assert np.float32(ent) == np.float32(rent.item())
    # and the oracle's values within the parity tolerances
    ref = oracle.forward(d["hidden"], d["weight"], d["targets"], bias=d["bias"], **c["kw"])
    assert_loss_close(loss if c["kw"]["reduction"] == "none" else loss[0], ref["loss"], "bf16")
    assert_lse_close(lse, ref["lse"])
    assert_entropy_close(ent, ref["entropy_sum"])


def test_noalloc_forward_matches_workspace_forward_twice():
    for c in CASES:   # two calls in a row on different inputs and options
        d, p, dev = setup(c)
        got = noalloc_forward(p, *dev)
        check_against_workspace_forward_and_oracle(c, d, p, dev, got)


def test_noalloc_expired_wait_gives_nan_not_stale_results():
    c = CASES[0]
    d, p, dev = setup(c)
    good = noalloc_forward(p, *dev)        # leaves this call's partial states in the array
    _lib.test_fault(1, 100)                # starve one stage; every wait gives up after 100 ms
    try:
        loss, lse, nc, ent = noalloc_forward(p, *dev)
    finally:
        _lib.test_fault(-1, 0)
    assert np.isnan(loss).all() and np.isnan(lse).all(), (loss, good[0])
    assert nc == -1 and np.isnan(ent)
    # the next call on the same process and array is correct again
    check_against_workspace_forward_and_oracle(c, d, p, dev, noalloc_forward(p, *dev))


def test_noalloc_rejects_sizes_beyond_the_fixed_scratch():
    p = _lib.make_params(N=65536, H=4096, V=128256, dtype=_lib.FLCE_BF16)
    assert _lib.workspace_bytes(p, _lib.FLCE_PASS_FORWARD) > SCRATCH_MAX
    n0 = _lib.launch_count()
    fake = 1 << 20   # never dereferenced: the size check comes first
    rc = _lib.forward_noalloc_raw(p, fake, fake, 0, fake, fake, fake, 0, 0, 0)
    assert rc == 4   # FLCE_ERR_WORKSPACE
    assert "fixed maximum" in _lib.last_error_detail()
    assert _lib.launch_count() == n0
