"""fp64 CPU oracle for the generic chunked linear loss. TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference leg
may import this module. The product path never imports or calls it, and it
shares no code with that path.

"Chunked Linear Loss" (sections "Why chunk the projection?" and "Loss function
contract") defines the strategy for ``logits = inputs @ weight.T`` followed by
a loss that is additive over rows. For each row chunk [r0, r1):

    Z_c          = X[r0:r1] W^T                      (the chunk's logits)
    (l_c, G_c)   = loss_and_grad(Z_c, sliced args)   (scalar loss, dL/dZ_c)
    dX[r0:r1]    = G_c W
    dW          += G_c^T X[r0:r1]

and the loss is sum_c l_c. Per-row tensor arguments (first dimension equal to
the number of rows of X) are sliced to the chunk ("Sliced arguments"); other
arguments pass through. Everything here is fp64; the one library primitive is
the matrix product. The chunking is kept exactly as the page states it, so a
reader can check each step; for an additive loss the result does not depend
on the chunk size (pinned).

The two losses below are written from their definitions.
- weighted_mse: the row- and feature-weighted squared error that the page uses
  as its direct-gradient example ("Direct logits gradients"):
      L = sum_ij r_i f_j (z_ij - y_ij)^2,   dL/dz_ij = 2 r_i f_j (z_ij - y_ij)
- cross_entropy_sum: summed softmax cross-entropy over rows whose target is
  not ignore_index:
      L = sum_i (lse_i - z_{i,t_i}),        dL/dz_ij = p_ij - [j == t_i]
  and 0 for ignored rows.

Pinned by tests/test_chunked_oracle_pins.py: torch fp64 autograd of the
unchunked losses, central finite differences, independence from the chunk
size, the W = 0 closed form, and agreement with the cross-entropy oracle.
"""
from __future__ import annotations

from typing import Callable, Optional

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def weighted_mse(z: np.ndarray, target, row_weight, feature_weight):
    """(sum_ij r_i f_j (z_ij - y_ij)^2, its gradient in z).

    With the residual d = z - y, the gradient is G = 2 r_i f_j d_ij, and the
    loss is half the elementwise product of G with d, summed.
    """
    d = _f64(z) - _f64(target)
    G = 2.0 * np.outer(_f64(row_weight), _f64(feature_weight)) * d
    return 0.5 * float(np.einsum("ij,ij->", G, d)), G


def cross_entropy_sum(z: np.ndarray, targets, ignore_index: int = -100):
    """(sum over valid rows of lse_i - z_{i,t_i}, its gradient in z)."""
    z = _f64(z)
    t = np.asarray(targets)
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    s = e.sum(axis=1, keepdims=True)
    lse = (m + np.log(s))[:, 0]
    p = e / s
    valid = t != ignore_index
    rows = np.nonzero(valid)[0]
    loss = float((lse[rows] - z[rows, t[rows]]).sum())
    g = np.where(valid[:, None], p, 0.0)
    g[rows, t[rows]] -= 1.0
    return loss, g


def _slice(a, n_rows: int, r0: int, r1: int):
    if isinstance(a, np.ndarray) and a.ndim >= 1 and a.shape[0] == n_rows:
        return a[r0:r1]
    return a


def chunked_linear_loss(inputs, weight, loss_and_grad: Callable, *args,
                        chunk_rows: Optional[int] = None, **kwargs):
    """Returns (loss, grad_inputs, grad_weight), all fp64."""
    X = _f64(inputs)
    W = _f64(weight)
    N = X.shape[0]
    rows = chunk_rows or max(N, 1)
    loss = 0.0
    dX = np.zeros_like(X)
    dW = np.zeros_like(W)
    for r0 in range(0, N, rows):
        r1 = min(N, r0 + rows)
        Z = X[r0:r1] @ W.T
        a = [_slice(v, N, r0, r1) for v in args]
        k = {key: _slice(v, N, r0, r1) for key, v in kwargs.items()}
        l_c, G = loss_and_grad(Z, *a, **k)
        G = _f64(G)
        loss += float(l_c)
        dX[r0:r1] = G @ W
        dW += G.T @ X[r0:r1]
    return loss, dX, dW
