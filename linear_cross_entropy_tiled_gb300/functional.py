"""PyTorch-facing API over the C ABI. PyTorch supplies device memory and streams only.

``fused_linear_cross_entropy`` mirrors the signature printed in the
fused-linear-ce README ("Full signature"). It adds ``z_loss_multiplier`` from
"Chunked Linear Cross-Entropy" ("Usage") and ``deterministic`` (accepted; every
reduction in the library is already in fixed order). Loss, lse and gradients
come from the library's CUDA kernels through ``flce_forward`` and
``flce_backward``. This module only checks shapes and dtypes, allocates
outputs and workspaces with torch, and passes pointers.
"""
from __future__ import annotations

import os
from typing import Optional

import torch

from . import _lib

_DTYPES = {torch.float32: _lib.FLCE_F32, torch.bfloat16: _lib.FLCE_BF16,
           torch.float16: _lib.FLCE_F16}
_CHECK = os.environ.get("FLCE_CHECK", "0") not in ("", "0")


def _ptr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _prepare(hidden, weight, targets, bias):
    if not (hidden.is_cuda and weight.is_cuda and targets.is_cuda):
        raise ValueError("hidden, weight and targets must be CUDA tensors (there is no CPU path)")
    if hidden.dtype not in _DTYPES:
        raise TypeError(f"hidden must be float32, bfloat16 or float16, got {hidden.dtype}")
    if weight.dtype != hidden.dtype or (bias is not None and bias.dtype != hidden.dtype):
        raise TypeError("weight and bias must have the dtype of hidden")
    H = hidden.shape[-1]
    if weight.dim() != 2 or weight.shape[1] != H:
        raise ValueError(f"weight must be [V, {H}], got {tuple(weight.shape)}")
    h2 = hidden.reshape(-1, H).contiguous()
    t1 = targets.reshape(-1).to(torch.int64).contiguous()
    if t1.shape[0] != h2.shape[0]:
        raise ValueError("targets must have one entry per row of hidden")
    w = weight.contiguous()
    b = bias.contiguous() if bias is not None else None
    if b is not None and b.shape != (w.shape[0],):
        raise ValueError(f"bias must be [V]={w.shape[0]}, got {tuple(b.shape)}")
    return h2, w, t1, b


def _params(h2, w, b, reduction, ignore_index, logit_scale, softcap, z_loss_multiplier,
            deterministic):
    return _lib.make_params(N=h2.shape[0], H=h2.shape[1], V=w.shape[0], dtype=_DTYPES[h2.dtype],
                            reduction=reduction, ignore_index=int(ignore_index),
                            logit_scale=float(logit_scale), softcap=softcap,
                            z_loss_multiplier=float(z_loss_multiplier), has_bias=b is not None,
                            deterministic=deterministic)


def _maybe_check(ws: torch.Tensor, where: str) -> None:
    if _CHECK:
        _lib.check(_lib.check_status(ws.data_ptr(), _stream(ws.device)), where)


def flce_forward(p: _lib.FlceParams, hidden: torch.Tensor, weight: torch.Tensor,
                 targets: torch.Tensor, bias: Optional[torch.Tensor] = None,
                 return_metrics: bool = False, workspace: Optional[torch.Tensor] = None):
    """One call of the C ABI forward on already-prepared contiguous tensors.

    Returns (loss, lse, num_correct or None, entropy_sum or None, workspace).
    """
    dev = hidden.device
    nloss = p.N if p.reduction == _lib.FLCE_NONE else 1
    loss = torch.empty(nloss, dtype=torch.float32, device=dev)
    lse = torch.empty(p.N, dtype=torch.float32, device=dev)
    nc = torch.empty(1, dtype=torch.int64, device=dev) if return_metrics else None
    ent = torch.empty(1, dtype=torch.float32, device=dev) if return_metrics else None
    need = _lib.workspace_bytes(p, _lib.FLCE_PASS_FORWARD)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    rc = _lib.forward_raw(p, _ptr(hidden), _ptr(weight), _ptr(bias), _ptr(targets), _ptr(loss),
                          _ptr(lse), _ptr(nc), _ptr(ent), _ptr(workspace), workspace.numel(),
                          _stream(dev))
    _lib.check(rc, "flce_forward")
    _maybe_check(workspace, "flce_forward")
    return loss, lse, nc, ent, workspace


def flce_forward_partial(p: _lib.FlceParams, hidden: torch.Tensor, weight_shard: torch.Tensor,
                         targets: torch.Tensor, bias_shard: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The vocabulary sweep of one shard. Returns its per-row states as a [N, 5] int32 tensor.

    Its 20-byte rows are ``flce_row_state``. Gather the states of every shard
    (for example with an all-gather) and pass them to ``flce_forward_combine``.
    """
    dev = hidden.device
    states = torch.empty((p.N, 5), dtype=torch.int32, device=dev)
    need = _lib.workspace_bytes(p, _lib.FLCE_PASS_FORWARD)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    rc = _lib.forward_partial_raw(p, _ptr(hidden), _ptr(weight_shard), _ptr(bias_shard),
                                  _ptr(targets), _ptr(states), _ptr(workspace), workspace.numel(),
                                  _stream(dev))
    _lib.check(rc, "flce_forward_partial")
    _maybe_check(workspace, "flce_forward_partial")
    return states


def flce_forward_combine(p: _lib.FlceParams, states: torch.Tensor, targets: torch.Tensor,
                         return_metrics: bool = False,
                         workspace: Optional[torch.Tensor] = None):
    """Merges [R, N, 5] shard states (in vocabulary order). Returns (loss, lse, num_correct, entropy_sum)."""
    dev = targets.device
    R = states.shape[0]
    states = states.contiguous()
    nloss = p.N if p.reduction == _lib.FLCE_NONE else 1
    loss = torch.empty(nloss, dtype=torch.float32, device=dev)
    lse = torch.empty(p.N, dtype=torch.float32, device=dev)
    nc = torch.empty(1, dtype=torch.int64, device=dev) if return_metrics else None
    ent = torch.empty(1, dtype=torch.float32, device=dev) if return_metrics else None
    need = _lib.workspace_bytes(p, _lib.FLCE_PASS_FORWARD)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    rc = _lib.forward_combine_raw(p, _ptr(states), R, _ptr(targets), _ptr(loss), _ptr(lse),
                                  _ptr(nc), _ptr(ent), _ptr(workspace), workspace.numel(),
                                  _stream(dev))
    _lib.check(rc, "flce_forward_combine")
    _maybe_check(workspace, "flce_forward_combine")
    return loss, lse, nc, ent


def flce_backward(p: _lib.FlceParams, hidden: torch.Tensor, weight: torch.Tensor,
                  targets: torch.Tensor, lse: torch.Tensor, grad_loss: torch.Tensor,
                  bias: Optional[torch.Tensor] = None, need_hidden: bool = True,
                  need_weight: bool = True, need_bias: bool = True,
                  workspace: Optional[torch.Tensor] = None, out=None, accumulate: bool = False):
    """One call of the C ABI backward. Returns (grad_hidden, grad_weight, grad_bias, workspace).

    ``out`` may pass preallocated (grad_hidden, grad_weight, grad_bias) tensors.
    With ``accumulate`` the gradients are added into ``out`` (beta = 1).
    """
    dev = hidden.device
    if accumulate:
        if out is None:
            raise ValueError("accumulate=True needs the out=(...) tensors to add into")
        p = _lib.FlceParams.from_buffer_copy(p)
        p.accumulate = 1
    if out is not None:
        gh, gw, gb = out
    else:
        gh = torch.empty_like(hidden) if need_hidden else None
        gw = torch.empty_like(weight) if need_weight else None
        gb = torch.empty_like(bias) if (need_bias and bias is not None) else None
    gl = grad_loss.to(device=dev, dtype=torch.float32).reshape(-1).contiguous()
    need = _lib.workspace_bytes(p, _lib.FLCE_PASS_BACKWARD)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    rc = _lib.backward_raw(p, _ptr(hidden), _ptr(weight), _ptr(bias), _ptr(targets), _ptr(lse),
                           _ptr(gl), _ptr(gh), _ptr(gw), _ptr(gb), _ptr(workspace),
                           workspace.numel(), _stream(dev))
    _lib.check(rc, "flce_backward")
    _maybe_check(workspace, "flce_backward")
    return gh, gw, gb, workspace


class _FLCE(torch.autograd.Function):
    @staticmethod
    def forward(ctx, hidden, weight, bias, targets, opts):
        (reduction, ignore_index, logit_scale, softcap, z_loss, return_metrics,
         deterministic, accum_dtype, fuse_grad_accum) = opts
        shape = targets.shape
        h2, w, t1, b = _prepare(hidden, weight, targets, bias)
        p = _params(h2, w, b, reduction, ignore_index, logit_scale, softcap, z_loss,
                    deterministic)
        p.grad_weight_accum = _lib.ACCUM_DTYPES[accum_dtype]
        ctx.fuse_grad_accum = fuse_grad_accum
        ctx.weight = weight if fuse_grad_accum else None
        loss, lse, nc, ent, _ = flce_forward(p, h2, w, t1, b, return_metrics)
        ctx.save_for_backward(h2, w, t1, lse, b)
        ctx.p = p
        ctx.hidden_shape = hidden.shape
        ctx.mark_non_differentiable(lse)
        if nc is not None:
            ctx.mark_non_differentiable(nc, ent)
        out = loss.reshape(shape) if reduction == "none" else loss.reshape(())
        if nc is None:
            return out, None, None
        return out, nc.reshape(()), ent.reshape(())

    @staticmethod
    def backward(ctx, grad_loss, _g1=None, _g2=None):
        h2, w, t1, lse, b = ctx.saved_tensors
        weight = ctx.weight
        if ctx.fuse_grad_accum and ctx.needs_input_grad[1] and weight.grad is not None \
                and weight.grad.is_contiguous() and weight.grad.dtype == weight.dtype:
            # Add grad_weight straight into the existing weight.grad (beta = 1) and
            # return None for it, as quack's fused gradient accumulation does. The
            # other two gradients start from zero in the same call.
            gh = torch.zeros_like(h2) if ctx.needs_input_grad[0] else None
            gb = torch.zeros_like(b) if (b is not None and ctx.needs_input_grad[2]) else None
            flce_backward(ctx.p, h2, w, t1, lse, grad_loss, b, accumulate=True,
                          out=(gh, weight.grad, gb))
            gw = None
        else:
            gh, gw, gb, _ = flce_backward(
                ctx.p, h2, w, t1, lse, grad_loss, b, need_hidden=ctx.needs_input_grad[0],
                need_weight=ctx.needs_input_grad[1], need_bias=ctx.needs_input_grad[2])
        if gh is not None:
            gh = gh.reshape(ctx.hidden_shape)
        return gh, gw, gb, None, None


def fused_linear_cross_entropy(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                               bias: Optional[torch.Tensor] = None, ignore_index: int = -100,
                               logit_scale: float = 1.0, softcap: Optional[float] = None,
                               z_loss_multiplier: float = 0.0, reduction: str = "mean",
                               return_metrics: bool = False, deterministic: bool = False,
                               grad_weight_accum_dtype: str = "fp32",
                               fuse_grad_accum: bool = False):
    """Cross-entropy of ``hidden @ weight.T (+ bias)`` against ``targets``. The logits are never stored.

    Returns ``loss``, or ``(loss, {"num_correct_tokens", "entropy_sum"})``
    when ``return_metrics``. The metrics are int64 / float32 scalar sums over
    non-ignored rows (fused-linear-ce README, "Metrics for free"). hidden,
    weight and bias all receive gradients.

    ``grad_weight_accum_dtype`` selects the accumulator of grad_weight across
    row chunks ("Chunked Linear Loss", "Weight-gradient accumulation dtype"):
    "fp32" (default) or "weight". With ``fuse_grad_accum``, an existing
    ``weight.grad`` gets the gradient added in place by the backward kernel
    instead of a separate add.
    """
    if grad_weight_accum_dtype not in _lib.ACCUM_DTYPES:
        raise ValueError("grad_weight_accum_dtype must be 'fp32' or 'weight'")
    opts = (reduction, ignore_index, logit_scale, softcap, z_loss_multiplier, return_metrics,
            deterministic, grad_weight_accum_dtype, fuse_grad_accum)
    loss, nc, ent = _FLCE.apply(hidden, weight, bias, targets, opts)
    if return_metrics:
        return loss, {"num_correct_tokens": nc, "entropy_sum": ent}
    return loss
