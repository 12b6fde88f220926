"""Fused linear cross-entropy for GB300 (sm_103a).

The CUDA library libflce.so does all of the computation. Its C ABI is in
include/flce.h and ``_lib`` binds it with ctypes. ``functional`` wraps it for
PyTorch tensors and autograd. Importing this package loads nothing: the
library is loaded on the first call, and that call raises if it is missing.
"""
from .chunked import (  # noqa: F401
    autograd_loss_and_logits_grad, chunked_linear_loss, weighted_mse_loss,
)
from .functional import (  # noqa: F401
    flce_backward, flce_forward, flce_forward_combine, flce_forward_partial,
    fused_linear_cross_entropy,
)

__all__ = ["fused_linear_cross_entropy", "flce_forward", "flce_backward",
           "flce_forward_partial", "flce_forward_combine", "chunked_linear_loss",
           "autograd_loss_and_logits_grad", "weighted_mse_loss"]
