"""Kernels per call, and the in-kernel reductions that replaced separate launches.

* The forward's merge sums the block sums itself (its last block to finish),
  so a forward with rows launches the logit-tile kernel and the merge only.
* The backward's first kernel (the row coefficients) clears the workspace
  header and the fp32 tile counters, so the backward issues no memset.
* The fp32 path's K-split contraction adds its split partials to grad_hidden
  in the last split of each tile to finish, in split order, so no
  split-reduce kernel follows it; its counters are left zero for the next
  call, and repeated calls give the same bits.
"""
import pytest
import torch

import oracle
from linear_cross_entropy_tiled_gb300 import _lib
from linear_cross_entropy_tiled_gb300.functional import flce_backward, flce_forward
from linear_cross_entropy_tiled_gb300.workloads import small_case

from flce_check import assert_grad_close, assert_loss_close, to_device

pytestmark = pytest.mark.gpu

DT = {"bf16": _lib.FLCE_BF16, "f32": _lib.FLCE_F32}


def kernels_of(fn):
    torch.cuda.synchronize()
    n0 = _lib.launch_count()
    out = fn()
    torch.cuda.synchronize()
    return _lib.launch_count() - n0, out


@pytest.mark.parametrize("dtype,N,H,V,bias", [
    ("f32", 256, 512, 8192, False),   # the fp32 workload's sizes: 4 vocabulary chunks
    ("f32", 130, 72, 600, True),
    ("bf16", 600, 256, 4100, True),   # N < V: 2 vocabulary chunks
    ("bf16", 1200, 256, 600, True),   # N >= V: 2 row chunks of 768 and 432 rows
])
def test_kernels_per_call(dtype, N, H, V, bias):
    d = small_case(N, H, V, seed=3, dtype=dtype, bias=bias, ignore_frac=0.1)
    h, w, b, t = to_device(d, dtype)
    p = _lib.make_params(N=N, H=H, V=V, dtype=DT[dtype], has_bias=bias, reduction="sum")
    n_fwd, (loss, lse, _, _, _) = kernels_of(lambda: flce_forward(p, h, w, t, b))
    assert n_fwd == 2                         # logit tiles, merge (with the reduction)
    gl = torch.ones(1, device="cuda")
    n_bwd, _ = kernels_of(lambda: flce_backward(p, h, w, t, lse, gl, b))
    # vocabulary chunks (four on the fp32 path, two on the 16-bit path, whose
    # one dlogits copy holds half of the columns) or, with N >= V, two row
    # chunks of half of the rows: each dlogits and both contractions (one grid
    # on the fp32 path; no K split at V = 600); row coefficients first (and h
    # transposed on the 16-bit path), grad_bias's sum last
    if dtype == "f32":
        assert n_bwd == 1 + 2 * 4 + (1 if bias else 0)
    else:
        assert n_bwd == 2 + 3 * 2 + (1 if bias else 0)


def test_row_chunks_adding_fp32_accumulated_grad_weight_keep_two_copies():
    """Row chunks that add into existing gradients with fp32 accumulation: the
    fp32 grad_weight partial starts from the output in its [V, H] layout, so
    grad_weight reads a transposed dlogits copy and h is not transposed. Two
    copies of a quarter of the rows: 3 chunks of 512, 512 and 176 rows."""
    N, H, V = 1200, 256, 600
    d = small_case(N, H, V, seed=8, dtype="bf16", bias=True, ignore_frac=0.1)
    h, w, b, t = to_device(d, "bf16")
    p = _lib.make_params(N=N, H=H, V=V, dtype=_lib.FLCE_BF16, has_bias=True, reduction="mean")
    _, lse, _, _, _ = flce_forward(p, h, w, t, b)
    out = (torch.zeros_like(h), torch.zeros_like(w), torch.zeros_like(b))
    gl = torch.ones(1, device="cuda")
    n_bwd, _ = kernels_of(lambda: flce_backward(p, h, w, t, lse, gl, b, accumulate=True, out=out))
    assert n_bwd == 1 + 3 * 3 + 1
    rgh, rgw, rgb = oracle.backward(d["hidden"], d["weight"], d["targets"], bias=d["bias"],
                                    reduction="mean")
    assert_grad_close(out[0].float().cpu().numpy(), rgh, "bf16", "grad_hidden")
    assert_grad_close(out[1].float().cpu().numpy(), rgw, "bf16", "grad_weight")
    assert_grad_close(out[2].float().cpu().numpy(), rgb, "bf16", "grad_bias")


@pytest.mark.parametrize("N,H,V,axis", [
    (256, 512, 8192, "vocab"),    # grad_hidden: 32 tiles x 4 K splits per chunk
    (200, 136, 3000, "rows"),     # grad_hidden K = V split per row chunk
    (70, 64, 9000, "vocab"),      # ragged row tile, 4 K splits
])
def test_fp32_split_counters_reset_and_repeatable(N, H, V, axis):
    d = small_case(N, H, V, seed=N, dtype="f32", bias=False, ignore_frac=0.1)
    h, w, _, t = to_device(d, "f32")
    p = _lib.make_params(N=N, H=H, V=V, dtype=_lib.FLCE_F32, reduction="sum",
                         bwd_chunk_axis=axis, max_chunk=64 if axis == "rows" else 0)
    loss, lse, _, _, _ = flce_forward(p, h, w, t)
    ref = oracle.forward(d["hidden"], d["weight"], d["targets"], reduction="sum")
    assert_loss_close(loss.item(), ref["loss"], "f32")
    gl = torch.ones(1, device="cuda")
    ws = torch.full((_lib.workspace_bytes(p, _lib.FLCE_PASS_BACKWARD),), 0x7F, dtype=torch.uint8,
                    device="cuda")   # counters start as garbage: the first kernel clears them
    outs = []
    for _ in range(3):
        gh, gw, _, ws = flce_backward(p, h, w, t, lse, gl, workspace=ws)
        torch.cuda.synchronize()
        regions = {n: (o, s) for n, o, s in _lib.workspace_regions(p, _lib.FLCE_PASS_BACKWARD)}
        o, s = regions["tile_counters"]
        assert torch.count_nonzero(ws[o:o + s]).item() == 0
        assert _lib.check_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
        outs.append((gh.clone(), gw.clone()))
    for gh, gw in outs[1:]:
        assert torch.equal(gh, outs[0][0]) and torch.equal(gw, outs[0][1])
    rgh, rgw, _ = oracle.backward(d["hidden"], d["weight"], d["targets"], reduction="sum")
    assert_grad_close(outs[0][0].cpu().numpy(), rgh, "f32", "grad_hidden")
    assert_grad_close(outs[0][1].cpu().numpy(), rgw, "f32", "grad_weight")


def test_fp32_large_grids_one_group_and_persistent_loop():
    """fp32 at N=1200, H=136, V=20000 (vocabulary chunks of 5056 columns).

    The forward (1501 units) and dlogits (1501 tiles) grids exceed two blocks
    per SM, so they run the 128-thread single-group kernels; the two
    contractions (285 + 237 units) run on the persistent grid of two blocks
    per SM, each block taking several units. Everything against the oracle.
    """
    N, H, V = 1200, 136, 20000
    d = small_case(N, H, V, seed=11, dtype="f32", bias=True, ignore_frac=0.1)
    h, w, b, t = to_device(d, "f32")
    kw = dict(reduction="mean", z_loss_multiplier=1e-3, softcap=20.0)
    p = _lib.make_params(N=N, H=H, V=V, dtype=_lib.FLCE_F32, has_bias=True, **kw)
    loss, lse, _, _, _ = flce_forward(p, h, w, t, b)
    ref = oracle.forward(d["hidden"], d["weight"], d["targets"], bias=d["bias"], **kw)
    assert_loss_close(loss.item(), ref["loss"], "f32")
    gl = torch.ones(1, device="cuda")
    gh, gw, gb, ws = flce_backward(p, h, w, t, lse, gl, b)
    torch.cuda.synchronize()
    assert _lib.check_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    rgh, rgw, rgb = oracle.backward(d["hidden"], d["weight"], d["targets"], bias=d["bias"], **kw)
    assert_grad_close(gh.cpu().numpy(), rgh, "f32", "grad_hidden")
    assert_grad_close(gw.cpu().numpy(), rgw, "f32", "grad_weight")
    assert_grad_close(gb.cpu().numpy(), rgb, "f32", "grad_bias")


def test_profiling_records_per_kernel():
    """flce_profiling_read: per-kernel launch counts, durations, clocks and MMA wait shares.

    Two read epochs in a row: each read returns only the launches since the
    previous one, and the clock records (zeroed once per epoch) give a clock
    within the GPU's range for every tensor-core kernel.
    """
    N, H, V = 1024, 512, 9000
    d = small_case(N, H, V, seed=21, dtype="bf16", bias=True, ignore_frac=0.05)
    h, w, b, t = to_device(d, "bf16")
    p = _lib.make_params(N=N, H=H, V=V, dtype=_lib.FLCE_BF16, has_bias=True, reduction="mean")
    gl = torch.ones(1, device="cuda")
    _lib.profiling_read()   # drop anything pending
    for steps in (1, 3):
        _lib.profiling_enable(True)
        for _ in range(steps):
            loss, lse, _, _, _ = flce_forward(p, h, w, t, b)
            flce_backward(p, h, w, t, lse, gl, b)
        _lib.profiling_enable(False)
        recs = {r[0]: r for r in _lib.profiling_read()}
        # forward: tiles + merge; backward: row coefficients, h transposed,
        # 2 x (dlogits, two GEMMs), bias sums
        assert recs["flce_fwd_tc"][1] == steps and recs["flce_merge"][1] == steps
        assert recs["flce_transpose_hidden"][1] == steps
        assert recs["flce_dlogits_tc"][1] == 2 * steps
        assert recs["flce_grad_hidden_tc"][1] == 2 * steps
        assert recs["flce_grad_weight_tc"][1] == 2 * steps
        for name in ("flce_fwd_tc", "flce_dlogits_tc", "flce_grad_hidden_tc", "flce_grad_weight_tc"):
            _, n, ms, mhz, (w_ops, w_acc) = recs[name]
            assert ms > 0.0, name
            assert 300.0 < mhz < 2600.0, (name, mhz)
            assert 0.0 <= w_ops <= 1.0 and 0.0 <= w_acc <= 1.0, (name, w_ops, w_acc)
        assert recs["flce_merge"][3] == 0.0   # the small kernels keep no clock record
    assert _lib.profiling_read() == []
