"""Generic chunked linear loss: any row-separable loss of ``logits = inputs @ weight.T``.

This follows "Chunked Linear Loss" (sections "Why chunk the projection?",
"What is fused?", "Loss function contract", "Sliced arguments"). The rows are
processed in chunks, and for each chunk:

1. the library computes the chunk's logits (``flce_chunk_logits``, the tcgen05
   GEMM for bf16 / fp16, the SIMT GEMM for fp32);
2. the caller's ``loss_and_grad_fn`` turns them into a scalar loss and the
   logits gradient of the same shape;
3. the library folds that gradient into the chunk's rows of grad_input and
   into grad_weight (``flce_chunk_grads``). grad_weight is summed over the
   chunks in an fp32 partial, or in the weight dtype when
   ``grad_weight_accum_dtype="weight"``.

Only one chunk of logits exists at a time. The gradients are computed in the
forward call, as the strategy on the page does, and scaled by the incoming
gradient in the backward.

``loss_and_grad_fn`` is the caller's code and runs as the caller wrote it,
on the chunk's device tensors. Tensor arguments whose first dimension equals
the number of rows of ``inputs`` are sliced to the chunk's rows; all other
arguments are passed unchanged. The chunk losses are summed, so the loss must
be additive over rows ("Reduction semantics").

``weighted_mse_loss(target, row_weight, feature_weight)`` can stand in for a
callback. It is the page's weighted squared error ("Direct logits
gradients") computed on the device: steps 1 and 2 become one kernel
(``flce_chunk_weighted_mse``) whose epilogue applies the loss to the fp32
accumulator, so the chunk's logits are never written.
"""
from __future__ import annotations

from typing import Callable, Optional

import torch

from . import _lib
from .functional import _DTYPES, _maybe_check, _ptr, _stream

# Rows per chunk by default: the logits chunk is kept near 1 GiB.
_CHUNK_BYTES = 1 << 30


def _round8(x: int) -> int:
    return (x + 7) // 8 * 8


def default_chunk_rows(n_rows: int, vocab: int, elem_bytes: int) -> int:
    """Rows per chunk: a multiple of 256 whose logits chunk is at most about 1 GiB."""
    rows = _CHUNK_BYTES // max(1, _round8(vocab) * elem_bytes) // 256 * 256
    return max(1, min(n_rows, max(256, rows)))


def _slice_arg(a, n_rows: int, r0: int, r1: int):
    if isinstance(a, torch.Tensor) and a.dim() >= 1 and a.shape[0] == n_rows:
        return a[r0:r1]
    return a


class _WeightedMSE:
    """sum_rv r_r f_v (z_rv - y_rv)^2 over the rows, evaluated inside the projection's epilogue."""

    def __init__(self, target: torch.Tensor, row_weight: torch.Tensor,
                 feature_weight: torch.Tensor):
        if target.dim() != 2 or row_weight.dim() != 1 or feature_weight.dim() != 1:
            raise ValueError("target must be [N, V], row_weight [N] and feature_weight [V]")
        self.target = target.float()
        if self.target.stride(1) != 1 or self.target.stride(0) % 4 != 0 \
                or self.target.data_ptr() % 16 != 0:
            # the kernel reads rows of a 4-float-multiple stride, 16-byte aligned
            N, V = self.target.shape
            padded = torch.empty((N, (V + 3) // 4 * 4), dtype=torch.float32,
                                 device=self.target.device)
            padded[:, :V].copy_(self.target)
            self.target = padded[:, :V]
        self.row_weight = row_weight.float().contiguous()
        self.feature_weight = feature_weight.float().contiguous()


def weighted_mse_loss(target: torch.Tensor, row_weight: torch.Tensor,
                      feature_weight: torch.Tensor) -> _WeightedMSE:
    """The weighted squared error as a device-side loss for ``chunked_linear_loss``."""
    return _WeightedMSE(target, row_weight, feature_weight)


class _ChunkedLinearLoss(torch.autograd.Function):
    @staticmethod
    def forward(ctx, inputs, weight, fn, opts):
        chunk_rows, accum, loss_args, loss_kwargs = opts
        if not (inputs.is_cuda and weight.is_cuda):
            raise ValueError("inputs and weight must be CUDA tensors (there is no CPU path)")
        if inputs.dtype not in _DTYPES or weight.dtype != inputs.dtype:
            raise TypeError("inputs and weight must share one of float32, bfloat16, float16")
        H = inputs.shape[-1]
        if weight.dim() != 2 or weight.shape[1] != H:
            raise ValueError(f"weight must be [V, {H}], got {tuple(weight.shape)}")
        x = inputs.reshape(-1, H).contiguous()
        w = weight.contiguous()
        N, V = x.shape[0], w.shape[0]
        dev = x.device
        need_x, need_w = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        gx = torch.empty_like(x) if need_x else None
        gw = torch.empty_like(w) if need_w else None
        total = torch.zeros((), dtype=torch.float32, device=dev)
        if N == 0:
            if gw is not None:
                gw.zero_()
            ctx.save_for_backward(gx, gw)
            ctx.shape = inputs.shape
            return total
        elem = x.element_size()
        rows = chunk_rows or default_chunk_rows(N, V, elem)
        rows = max(1, min(int(rows), N))
        nchunks = -(-N // rows)
        ld = _round8(V)
        dtype = _DTYPES[x.dtype]
        kw = dict(H=H, V=V, dtype=dtype, grad_weight_accum=accum)
        p_max = _lib.make_params(N=rows, **kw)
        logits = torch.empty((rows, ld), dtype=x.dtype, device=dev)
        ws_l = torch.empty(max(256, _lib.workspace_bytes(p_max, _lib.FLCE_PASS_CHUNK_LOGITS)),
                           dtype=torch.uint8, device=dev)
        ws_g = torch.empty(max(256, _lib.workspace_bytes(p_max, _lib.FLCE_PASS_CHUNK_GRADS)),
                           dtype=torch.uint8, device=dev)
        staged = None
        stream = _stream(dev)
        device_loss = isinstance(fn, _WeightedMSE)
        if device_loss:
            if fn.target.shape != (N, V) or fn.row_weight.shape != (N,) or \
                    fn.feature_weight.shape != (V,):
                raise ValueError("weighted_mse_loss: target [N, V], row_weight [N], "
                                 "feature_weight [V] must match inputs and weight")
            loss64 = torch.zeros(1, dtype=torch.float64, device=dev)
            # no transposed dlogits copy: flce_chunk_grads computes grad_weight
            # transposed, from h^T and the row-major dlogits
            ws_m = torch.empty(max(256, _lib.workspace_bytes(p_max, _lib.FLCE_PASS_CHUNK_MSE)),
                               dtype=torch.uint8, device=dev)
        for c in range(nchunks):
            r0, r1 = c * rows, min(N, (c + 1) * rows)
            p = _lib.make_params(N=r1 - r0, **kw)
            xc = x[r0:r1]
            if device_loss:
                # steps 1 and 2 in one kernel: the logits never leave the accumulator
                tgt = fn.target[r0:r1]
                rc = _lib.chunk_weighted_mse_raw(
                    p, _ptr(xc), _ptr(w), _ptr(tgt), tgt.stride(0), _ptr(fn.row_weight[r0:r1]),
                    _ptr(fn.feature_weight), _ptr(logits), ld, _ptr(loss64), 1 if c > 0 else 0,
                    _ptr(ws_m), ws_m.numel(), stream, 0, 0)
                _lib.check(rc, "flce_chunk_weighted_mse")
                _maybe_check(ws_m, "flce_chunk_weighted_mse")
                g = logits[: r1 - r0]
            else:
                _lib.check(_lib.chunk_logits_raw(p, _ptr(xc), _ptr(w), _ptr(logits), ld,
                                                 _ptr(ws_l), ws_l.numel(), stream),
                           "flce_chunk_logits")
                _maybe_check(ws_l, "flce_chunk_logits")
                args = [_slice_arg(a, N, r0, r1) for a in loss_args]
                kwargs = {k: _slice_arg(a, N, r0, r1) for k, a in loss_kwargs.items()}
                loss_c, g = fn(logits[: r1 - r0, :V], *args, **kwargs)
                if loss_c.dim() != 0:
                    raise ValueError("loss_and_grad_fn must return a scalar loss")
                total += loss_c.float()
            if not (need_x or need_w):
                continue
            if device_loss:
                pass   # g is the kernel's own [rows][ld] buffer
            elif g.shape != (r1 - r0, V):
                raise ValueError(f"the logits gradient must be [{r1 - r0}, {V}], got {tuple(g.shape)}")
            g = g.to(x.dtype)
            ok = (g.stride(1) == 1 and g.stride(0) >= V and g.stride(0) % 8 == 0
                  and g.data_ptr() % 16 == 0) or device_loss
            if not ok:
                # The kernels read rows of 16-byte-aligned, 8-element-multiple
                # stride; anything else is copied into a buffer of that layout.
                if staged is None:
                    staged = torch.empty((rows, ld), dtype=x.dtype, device=dev)
                staged[: r1 - r0, :V].copy_(g)
                g = staged[: r1 - r0]
            phase = (_lib.FLCE_CHUNK_ONLY if nchunks == 1 else _lib.FLCE_CHUNK_FIRST if c == 0
                     else _lib.FLCE_CHUNK_LAST if c == nchunks - 1 else _lib.FLCE_CHUNK_NEXT)
            rc = _lib.chunk_grads_raw(p, _ptr(xc), _ptr(w), _ptr(g), g.stride(0), phase,
                                      _ptr(gx[r0:r1]) if gx is not None else 0, _ptr(gw),
                                      _ptr(ws_g), ws_g.numel(), stream, 0, 0)
            _lib.check(rc, "flce_chunk_grads")
            _maybe_check(ws_g, "flce_chunk_grads")
        if device_loss:
            total = loss64[0].float()
        ctx.save_for_backward(gx, gw)
        ctx.shape = inputs.shape
        return total

    @staticmethod
    def backward(ctx, grad_out):
        # The gradients computed in the forward, times the upstream scalar
        # ("Gradient handling"), by the library's scale kernel. It writes new
        # tensors, so a second backward (retain_graph) still starts from the
        # unscaled ones.
        gx, gw = ctx.saved_tensors
        g = grad_out.to(dtype=torch.float32).reshape(1).contiguous()
        out = []
        for t in (gx, gw):
            if t is None:
                out.append(None)
                continue
            o = torch.empty_like(t)
            _lib.check(_lib.scale_raw(_ptr(t), _ptr(o), t.numel(), _DTYPES[t.dtype], _ptr(g),
                                      _stream(t.device)), "flce_scale")
            out.append(o)
        gx, gw = out
        if gx is not None:
            gx = gx.reshape(ctx.shape)
        return gx, gw, None, None


def chunked_linear_loss(inputs: torch.Tensor, weight: torch.Tensor,
                        loss_and_grad_fn: Callable, *loss_args,
                        chunk_rows: Optional[int] = None, grad_weight_accum_dtype: str = "fp32",
                        **loss_kwargs) -> torch.Tensor:
    """Sum over row chunks of ``loss_and_grad_fn(inputs[chunk] @ weight.T, *sliced args)[0]``.

    ``loss_and_grad_fn(logits_chunk, *args, **kwargs)`` returns
    ``(scalar loss, grad_logits)``, with grad_logits of the chunk's shape.
    Only ``inputs`` and ``weight`` receive gradients.

    ``chunk_rows`` defaults to a multiple of 256 with a logits chunk of about
    1 GiB. ``grad_weight_accum_dtype`` picks the accumulator of grad_weight
    across chunks: "fp32" (default) or "weight".
    """
    if grad_weight_accum_dtype not in _lib.ACCUM_DTYPES:
        raise ValueError("grad_weight_accum_dtype must be 'fp32' or 'weight'")
    opts = (chunk_rows, grad_weight_accum_dtype, loss_args, loss_kwargs)
    return _ChunkedLinearLoss.apply(inputs, weight, loss_and_grad_fn, opts)


def autograd_loss_and_logits_grad(loss_fn: Callable) -> Callable:
    """Adapts a loss that returns only a scalar ("Adapting PyTorch losses").

    The gradient of the loss in the logits chunk comes from PyTorch's
    functional transform ``torch.func.grad_and_value``, applied to the loss
    with the chunk's other arguments fixed. Returns ``(loss, d loss / d logits)``.
    """
    from torch.func import grad_and_value

    def fn(logits, *args, **kwargs):
        g, loss = grad_and_value(lambda z: loss_fn(z, *args, **kwargs))(logits.detach())
        return loss.detach(), g
    return fn
