"""GPU parity of the generic chunked linear loss ("Chunked Linear Loss") against the fp64 oracle.

The projection of each chunk (flce_chunk_logits) and the folding of the
caller's logits gradient into grad_input and grad_weight (flce_chunk_grads)
run in the library's kernels. The loss callbacks below are the caller's code,
written in torch as a user of the strategy would write them. They see the
chunk's logits in the input dtype, so the bar is the 16-bit one from
flce_check (fp32 for fp32 inputs).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from linear_cross_entropy_tiled_gb300 import autograd_loss_and_logits_grad, chunked_linear_loss
from linear_cross_entropy_tiled_gb300.workloads import round_to_16bit

from flce_check import TOL, assert_grad_close

pytestmark = pytest.mark.gpu

TDT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def stored(x, dtype):
    """(values the GPU holds as float64, device tensor)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x.astype(np.float64), torch.from_numpy(x).cuda()
    bits, vals = round_to_16bit(x, dtype)
    return vals.astype(np.float64), torch.from_numpy(bits.view(np.int16)).cuda().view(TDT[dtype])


def case(N, H, V, dtype, seed):
    g = np.random.default_rng(seed)
    X, Xd = stored(g.standard_normal((N, H)), dtype)
    W, Wd = stored(g.standard_normal((V, H)) / np.sqrt(H), dtype)
    Y = g.standard_normal((N, V)).astype(np.float32)
    r = g.uniform(0.5, 1.5, N).astype(np.float32)
    f = g.uniform(0.5, 1.5, V).astype(np.float32)
    return X, W, Y, r, f, Xd, Wd


def wmse_torch(z, y, rw, fw):
    """The caller's weighted MSE: loss and logits gradient from one chunk of logits.

    grad = 2 r f (z - y); the loss is half the dot product of grad with the residual.
    """
    d = torch.sub(z.float(), y)
    grad = torch.outer(rw, fw).mul_(d).mul_(2.0)
    return 0.5 * torch.dot(grad.flatten(), d.flatten()), grad.to(z.dtype)


def run(Xd, Wd, Y, r, f, **kw):
    x = Xd.clone().requires_grad_(True)
    w = Wd.clone().requires_grad_(True)
    loss = chunked_linear_loss(x, w, wmse_torch, torch.from_numpy(Y).cuda(),
                               torch.from_numpy(r).cuda(), torch.from_numpy(f).cuda(), **kw)
    loss.backward()
    torch.cuda.synchronize()
    return float(loss.item()), x.grad.double().cpu().numpy(), w.grad.double().cpu().numpy()


@pytest.mark.parametrize("dtype,N,H,V,chunk_rows,accum", [
    ("bf16", 1000, 264, 700, 256, "fp32"),    # 4 chunks, ragged rows, V and H
    ("bf16", 300, 128, 520, None, "fp32"),    # one chunk
    ("bf16", 700, 136, 900, 256, "weight"),   # grad_weight accumulated in bf16
    ("f16", 600, 200, 640, 256, "fp32"),
    ("f32", 300, 72, 500, 128, "fp32"),       # the SIMT path
])
def test_weighted_mse_matches_the_oracle(dtype, N, H, V, chunk_rows, accum):
    X, W, Y, r, f, Xd, Wd = case(N, H, V, dtype, seed=N + V)
    loss, gx, gw = run(Xd, Wd, Y, r, f, chunk_rows=chunk_rows, grad_weight_accum_dtype=accum)
    ref, rx, rw = oracle.chunked_linear_loss(X, W, oracle.weighted_mse, Y, r, f,
                                             chunk_rows=chunk_rows)
    assert abs(loss - ref) <= TOL[dtype]["loss"] * abs(ref), (loss, ref)
    assert_grad_close(gx, rx, dtype, "grad_inputs")
    assert_grad_close(gw, rw, dtype, "grad_weight")


def test_cross_entropy_through_the_autograd_adapter_matches_the_fused_oracle():
    N, H, V = 700, 256, 1100
    X, W, _, _, _, Xd, Wd = case(N, H, V, "bf16", seed=5)
    t = np.random.default_rng(6).integers(0, V, N)
    t[::7] = -100
    fn = autograd_loss_and_logits_grad(
        lambda z, tt: F.cross_entropy(z.float(), tt, ignore_index=-100, reduction="sum"))
    x = Xd.clone().requires_grad_(True)
    w = Wd.clone().requires_grad_(True)
    loss = chunked_linear_loss(x, w, fn, torch.from_numpy(t).cuda(), chunk_rows=256)
    loss.backward()
    torch.cuda.synchronize()
    ref = oracle.forward(X, W, t, reduction="sum")
    rx, rw, _ = oracle.backward(X, W, t, reduction="sum")
    assert abs(loss.item() - ref["loss"]) <= TOL["bf16"]["loss"] * abs(ref["loss"])
    assert_grad_close(x.grad.double().cpu().numpy(), rx, "bf16", "grad_inputs")
    assert_grad_close(w.grad.double().cpu().numpy(), rw, "bf16", "grad_weight")


def test_strided_logits_gradient_and_scaled_backward():
    """A callback gradient in column-major layout is staged; d(3 L) scales both gradients."""
    N, H, V = 520, 96, 333
    X, W, Y, r, f, Xd, Wd = case(N, H, V, "bf16", seed=9)

    def fn(z, y, rw, fw):
        loss, g = wmse_torch(z, y, rw, fw)
        return loss, g.t().contiguous().t()   # same values, column-major strides

    x = Xd.clone().requires_grad_(True)
    w = Wd.clone().requires_grad_(True)
    loss = chunked_linear_loss(x, w, fn, torch.from_numpy(Y).cuda(), torch.from_numpy(r).cuda(),
                               torch.from_numpy(f).cuda(), chunk_rows=256)
    (3.0 * loss).backward()
    torch.cuda.synchronize()
    ref, rx, rw = oracle.chunked_linear_loss(X, W, oracle.weighted_mse, Y, r, f, chunk_rows=256)
    assert abs(loss.item() - ref) <= TOL["bf16"]["loss"] * abs(ref)
    assert_grad_close(x.grad.double().cpu().numpy(), 3.0 * rx, "bf16", "grad_inputs")
    assert_grad_close(w.grad.double().cpu().numpy(), 3.0 * rw, "bf16", "grad_weight")


@pytest.mark.parametrize("dtype,N,H,V,chunk_rows", [
    ("bf16", 1000, 264, 700, 256),   # 4 chunks; 700 is not a multiple of 8
    ("bf16", 600, 128, 701, 256),    # V not a multiple of 4: the target is padded
    ("f16", 520, 200, 512, None),    # one chunk
])
def test_device_weighted_mse_matches_the_oracle(dtype, N, H, V, chunk_rows):
    """weighted_mse_loss: the loss inside the projection's epilogue (flce_chunk_weighted_mse)."""
    from linear_cross_entropy_tiled_gb300 import weighted_mse_loss
    X, W, Y, r, f, Xd, Wd = case(N, H, V, dtype, seed=3 * N + V)
    x = Xd.clone().requires_grad_(True)
    w = Wd.clone().requires_grad_(True)
    loss_fn = weighted_mse_loss(torch.from_numpy(Y).cuda(), torch.from_numpy(r).cuda(),
                                torch.from_numpy(f).cuda())
    loss = chunked_linear_loss(x, w, loss_fn, chunk_rows=chunk_rows)
    loss.backward()
    torch.cuda.synchronize()
    ref, rx, rw = oracle.chunked_linear_loss(X, W, oracle.weighted_mse, Y, r, f,
                                             chunk_rows=chunk_rows)
    # the loss is taken from the fp32 accumulator, so it is closer than the 16-bit bar
    assert abs(loss.item() - ref) <= 1e-4 * abs(ref), (loss.item(), ref)
    assert_grad_close(x.grad.double().cpu().numpy(), rx, dtype, "grad_inputs")
    assert_grad_close(w.grad.double().cpu().numpy(), rw, dtype, "grad_weight")
    # the same loss through the torch callback path
    loss2, gx2, gw2 = run(Xd, Wd, Y, r, f, chunk_rows=chunk_rows)
    assert abs(loss2 - loss.item()) <= TOL[dtype]["loss"] * abs(ref)
    assert_grad_close(x.grad.double().cpu().numpy(), gx2, dtype, "device vs callback grad_inputs")


def test_device_weighted_mse_refuses_fp32_inputs():
    from linear_cross_entropy_tiled_gb300 import weighted_mse_loss
    X, W, Y, r, f, Xd, Wd = case(64, 32, 48, "f32", seed=1)
    loss_fn = weighted_mse_loss(torch.from_numpy(Y).cuda(), torch.from_numpy(r).cuda(),
                                torch.from_numpy(f).cuda())
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        chunked_linear_loss(Xd.requires_grad_(True), Wd.requires_grad_(True), loss_fn)


@pytest.mark.parametrize("dtype,N,H,V,chunk_rows", [
    ("bf16", 3, 8, 5, None),      # every tile ragged; no 3-D view (fewer than two 64-column atoms)
    ("bf16", 7, 72, 130, 1),      # one-row chunks: FIRST, six NEXT, LAST
    ("f32", 5, 3, 7, 2),          # the SIMT path with odd sizes
])
def test_tiny_and_ragged_chunks(dtype, N, H, V, chunk_rows):
    X, W, Y, r, f, Xd, Wd = case(N, H, V, dtype, seed=N * 31 + V)
    loss, gx, gw = run(Xd, Wd, Y, r, f, chunk_rows=chunk_rows)
    ref, rx, rw = oracle.chunked_linear_loss(X, W, oracle.weighted_mse, Y, r, f,
                                             chunk_rows=chunk_rows)
    assert abs(loss - ref) <= TOL[dtype]["loss"] * abs(ref) + 1e-6, (loss, ref)
    assert_grad_close(gx, rx, dtype, "grad_inputs")
    assert_grad_close(gw, rw, dtype, "grad_weight")


@pytest.mark.parametrize("which", ["inputs", "weight"])
def test_gradient_of_one_argument_only(which):
    N, H, V = 400, 128, 600
    X, W, Y, r, f, Xd, Wd = case(N, H, V, "bf16", seed=21)
    x = Xd.clone().requires_grad_(which == "inputs")
    w = Wd.clone().requires_grad_(which == "weight")
    loss = chunked_linear_loss(x, w, wmse_torch, torch.from_numpy(Y).cuda(),
                               torch.from_numpy(r).cuda(), torch.from_numpy(f).cuda(),
                               chunk_rows=256)
    loss.backward()
    torch.cuda.synchronize()
    ref, rx, rw = oracle.chunked_linear_loss(X, W, oracle.weighted_mse, Y, r, f, chunk_rows=256)
    if which == "inputs":
        assert w.grad is None
        assert_grad_close(x.grad.double().cpu().numpy(), rx, "bf16", "grad_inputs")
    else:
        assert x.grad is None
        assert_grad_close(w.grad.double().cpu().numpy(), rw, "bf16", "grad_weight")


@pytest.mark.parametrize("V", [20480, 19999])
@pytest.mark.parametrize("loss_kind", ["device", "callback"])
def test_grouped_tile_raster_matches_the_oracle(V, loss_kind):
    """The projection's grouped raster: more column tiles than CTA pairs.

    With V / 256 = 80 column tiles (79 for the ragged V = 19999) a wave of the
    at most 76 co-resident pairs of a GB300 spans fewer than all column tiles,
    so the plain GEMM rasters its tiles in groups of row tiles, column after
    column within a group. N = 1000 in one chunk gives a group of four row
    tiles, the last one ragged; chunks of 512 rows give groups of two. Both the
    device-side weighted squared error and the torch callback go through that
    projection; every element is compared with the oracle.
    """
    from linear_cross_entropy_tiled_gb300 import weighted_mse_loss
    N, H = 1000, 256
    X, W, Y, r, f, Xd, Wd = case(N, H, V, "bf16", seed=V + 13)
    for chunk_rows in (None, 512):
        if loss_kind == "device":
            x = Xd.clone().requires_grad_(True)
            w = Wd.clone().requires_grad_(True)
            fn = weighted_mse_loss(torch.from_numpy(Y).cuda(), torch.from_numpy(r).cuda(),
                                   torch.from_numpy(f).cuda())
            lt = chunked_linear_loss(x, w, fn, chunk_rows=chunk_rows)
            lt.backward()
            torch.cuda.synchronize()
            loss, gx, gw = float(lt.item()), x.grad.double().cpu().numpy(), w.grad.double().cpu().numpy()
        else:
            loss, gx, gw = run(Xd, Wd, Y, r, f, chunk_rows=chunk_rows)
        ref, rx, rw = oracle.chunked_linear_loss(X, W, oracle.weighted_mse, Y, r, f,
                                                 chunk_rows=chunk_rows)
        tol = 1e-4 if loss_kind == "device" else TOL["bf16"]["loss"]
        assert abs(loss - ref) <= tol * abs(ref), (chunk_rows, loss, ref)
        assert_grad_close(gx, rx, "bf16", f"grad_inputs (chunk_rows={chunk_rows})")
        assert_grad_close(gw, rw, "bf16", f"grad_weight (chunk_rows={chunk_rows})")
