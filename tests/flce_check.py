"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and compare it with the oracle.

Tolerances. The bf16 ones are the stated bar, applied to fp16 as well (fp16
carries more mantissa than bf16). The fp32 gradient bar follows from fp32
accumulation over K <= V terms: the error grows like sqrt(K) * 2^-24 relative
to the terms, about 1e-5 at K = 8192, so 1e-4 of the largest gradient. The lse
bar covers fp32 arithmetic with ex2.approx (relative error near 2^-22):
  loss          relative error <= 2e-3 (bf16 inputs), <= 1e-5 (fp32 inputs)
  lse           |err| <= 1e-4 * max(1, |lse|)  (fp32 arithmetic on both dtypes)
  gradients     max|err| <= 2e-2 * max|ref| and cosine >= 0.9999 (bf16);
                max|err| <= 1e-4 * max|ref| and cosine >= 0.999999 (fp32)
  num_correct   exact, except rows whose top-2 oracle logits lie within 1e-3
  entropy_sum   relative error <= 1e-3
"""
from __future__ import annotations

import numpy as np
import torch

from linear_cross_entropy_tiled_gb300 import _lib
from linear_cross_entropy_tiled_gb300.functional import flce_backward, flce_forward

TOL = {
    "bf16": dict(loss=2e-3, grad_max=2e-2, grad_cos=0.9999),
    "f16": dict(loss=2e-3, grad_max=2e-2, grad_cos=0.9999),
    "f32": dict(loss=1e-5, grad_max=1e-4, grad_cos=0.999999),
}
NEAR_TIE = 1e-3


def to_device(d: dict, dtype: str, dev="cuda"):
    """Device tensors holding exactly the values the oracle reads."""
    def mat(name):
        if dtype in ("bf16", "f16"):
            bits = d[name + "_bits"]
            tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
            return torch.from_numpy(bits.view(np.int16)).to(dev).view(tdt)
        return torch.from_numpy(np.ascontiguousarray(d[name], dtype=np.float32)).to(dev)
    h = mat("hidden")
    w = mat("weight")
    b = mat("bias") if d.get("bias") is not None else None
    t = torch.from_numpy(d["targets"]).to(dev)
    return h, w, b, t


def run_gpu(d: dict, dtype: str, kw: dict, grad_loss=1.0, return_metrics=True,
            need=(True, True, True), schedule=None):
    """Forward + backward through the C ABI. Returns numpy outputs.

    ``schedule`` holds flce_params fields that change only how the backward is
    cut into chunks (bwd_chunk_axis, max_chunk), never the result.
    """
    h, w, b, t = to_device(d, dtype)
    dt = {"bf16": _lib.FLCE_BF16, "f16": _lib.FLCE_F16, "f32": _lib.FLCE_F32}[dtype]
    p = _lib.make_params(N=h.shape[0], H=h.shape[1], V=w.shape[0], dtype=dt,
                         has_bias=b is not None, **kw, **(schedule or {}))
    loss, lse, nc, ent, fws = flce_forward(p, h, w, t, b, return_metrics=return_metrics)
    st = _lib.check_status(fws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    gl = torch.as_tensor(np.asarray(grad_loss, dtype=np.float32).reshape(-1), device=h.device)
    gh, gw, gb, bws = flce_backward(p, h, w, t, lse, gl, b, need_hidden=need[0],
                                    need_weight=need[1], need_bias=need[2])
    st2 = _lib.check_status(bws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    f = lambda x: None if x is None else x.float().cpu().numpy()
    return dict(loss=f(loss), lse=f(lse), num_correct=None if nc is None else int(nc.item()),
                entropy_sum=None if ent is None else float(ent.item()), grad_hidden=f(gh),
                grad_weight=f(gw), grad_bias=f(gb), status_fwd=st, status_bwd=st2)


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


def assert_grad_close(got, ref, dtype, name):
    tol = TOL[dtype]
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    if scale == 0:
        assert err == 0, (name, err)
        return
    assert err <= tol["grad_max"] * scale, f"{name}: max err {err:.3e} vs {tol['grad_max']} * {scale:.3e}"
    c = cosine(got, ref)
    assert c >= tol["grad_cos"], f"{name}: cosine {c:.8f}"


def assert_loss_close(got, ref, dtype, name="loss"):
    tol = TOL[dtype]["loss"]
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.ndim == 0 or ref.size == 1:
        r = float(ref.reshape(-1)[0])
        g = float(got.reshape(-1)[0])
        if np.isnan(r):
            assert np.isnan(g), (name, g)
            return
        assert abs(g - r) <= tol * abs(r) + 1e-12, f"{name}: {g} vs {r}"
    else:
        # per-row losses: relative to the row, with an absolute floor of tol*mean
        floor = tol * max(np.abs(ref).mean(), 1e-30)
        err = np.abs(got - ref)
        assert (err <= tol * np.abs(ref) + floor).all(), f"{name}: max err {err.max():.3e}"


def assert_lse_close(got, ref, name="lse"):
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    lim = 1e-4 * np.maximum(1.0, np.abs(ref))
    assert (err <= lim).all(), f"{name}: max err {err.max():.3e}"


def assert_num_correct(got: int, ref_fwd_rows: dict, targets, ignore_index=-100):
    """Exact, except that rows whose top-2 oracle logits are within 1e-3 may go either way."""
    t = np.asarray(targets)
    valid = t != ignore_index
    near = ref_fwd_rows["top2_gap"] < NEAR_TIE
    sure = int((ref_fwd_rows["correct"] & ~near & valid).sum())
    unsure = int((near & valid).sum())
    assert sure <= got <= sure + unsure, (got, sure, unsure)


def assert_entropy_close(got, ref):
    assert abs(got - ref) <= 1e-3 * abs(ref) + 1e-9, (got, ref)
