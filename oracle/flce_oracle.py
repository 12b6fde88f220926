"""fp64 CPU oracle for fused linear cross-entropy. TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference leg
may import this module. The product path (the CUDA library and its Python
binding) never imports or calls it, and it shares no code with that path. The
only common module is the seeded input generator, which holds none of this
arithmetic.

What it computes is the plain definition. Every logit is materialised in fp64.
The one library primitive is the fp64 matrix product of the projection.

Projection and loss. quack-kernels diff, ``quack/linear_cross_entropy.py``,
``linear_cross_entropy_func_ref``: ``F.linear`` followed by ``F.cross_entropy``
with ``ignore_index`` and ``reduction``.

    a_ij   = sum_k h_ik W_jk

Logit transforms, in this order. fused-linear-ce README, sections "Full
signature" (``bias``, ``logit_scale``, ``softcap``) and "Algorithm" (the tile
"applies bias / logit_scale / softcap"):

    u_ij   = (a_ij + b_j) * s
    z_ij   = c * tanh(u_ij / c)   when a softcap c > 0 is given, else u_ij

Per valid row (t_i != ignore_index):

    lse_i  = log sum_j exp(z_ij)
    loss_i = lse_i - z_{i,t_i} + zeta * lse_i^2

The z-loss term is a reading. "Chunked Linear Cross-Entropy", section "Usage",
names only ``z_loss_multiplier``. It is taken as the usual zeta * lse^2 per
valid row, added into the same reduction. Ignored rows have loss 0.

Reductions ("Chunked Linear Loss", section "Reduction semantics"; the quack
diff, ``ChunkedLinearCrossEntropyFunction.forward``):
    sum  -> sum_i loss_i
    mean -> sum_i loss_i / (number of valid rows over the whole call)
    none -> the vector loss_i

Metrics (fused-linear-ce README, "Metrics for free"). Both are sums over valid
rows and carry no gradient.
    num_correct_tokens = #{valid i : argmax_j z_ij == t_i}   (ties: lowest j)
    entropy_sum        = sum_i (lse_i - sum_j p_ij z_ij),  p_ij = exp(z_ij - lse_i)

Gradients (fused-linear-ce README, "Algorithm": the backward forms p - onehot
and contracts it with W and with h; quack diff, the backward scales by dloss):

    g_ij = gamma_i * (p_ij * (1 + 2 zeta lse_i) - [j == t_i]) * (1 - (z_ij/c)^2) * s

The factor (1 - (z/c)^2) is present only with a softcap. gamma_i is grad_loss
for sum, grad_loss / num_valid for mean and grad_loss_i for none. It is 0 on
ignored rows.

    grad_hidden = g W,    grad_weight = g^T h,    grad_bias_j = sum_i g_ij

Every function below is pinned by tests/test_oracle_pins.py. The pins are
torch's fp64 autograd of ``F.cross_entropy(F.linear(...))``, central finite
differences, closed forms, invariants and hand-derived golden values.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

REDUCTIONS = ("sum", "mean", "none")


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def check_targets(targets: np.ndarray, V: int, ignore_index: int) -> None:
    """A target is either ignore_index or a class id in [0, V). Anything else is an error.

    F.cross_entropy in the quack reference raises on such a target.
    """
    t = np.asarray(targets)
    bad = (t != ignore_index) & ((t < 0) | (t >= V))
    if bad.any():
        raise ValueError(f"{int(bad.sum())} target(s) outside [0, {V}) and not ignore_index")


def transformed_logits(hidden, weight, bias=None, logit_scale: float = 1.0,
                       softcap: Optional[float] = None) -> np.ndarray:
    """z = softcap(((h W^T) + b) * s) in fp64, for the given rows of ``hidden``."""
    a = _f64(hidden) @ _f64(weight).T
    if bias is not None:
        a = a + _f64(bias)[None, :]
    u = a * float(logit_scale)
    if softcap is not None and softcap > 0:
        c = float(softcap)
        return c * np.tanh(u / c)
    return u


def row_terms(z: np.ndarray, targets: np.ndarray, ignore_index: int,
              z_loss_multiplier: float = 0.0) -> dict:
    """Per-row quantities of a block of fully materialised logit rows ``z`` [n, V]."""
    n = z.shape[0]
    t = np.asarray(targets, dtype=np.int64)
    valid = t != ignore_index
    m = z.max(axis=1)
    e = np.exp(z - m[:, None])
    ssum = e.sum(axis=1)
    lse = m + np.log(ssum)
    p = e / ssum[:, None]
    tsafe = np.where(valid, t, 0)
    zt = z[np.arange(n), tsafe]
    zeta = float(z_loss_multiplier)
    loss = np.where(valid, lse - zt + zeta * lse * lse, 0.0)
    entropy = lse - (p * z).sum(axis=1)
    argmax = z.argmax(axis=1)  # numpy returns the first index that attains the max
    correct = valid & (argmax == t)
    return dict(lse=lse, loss=loss, entropy=entropy, argmax=argmax, correct=correct,
                valid=valid, p=p, z=z)


def _reduce(loss_rows: np.ndarray, num_valid: int, reduction: str):
    if reduction == "sum":
        return float(loss_rows.sum())
    if reduction == "mean":
        return float(loss_rows.sum()) / num_valid if num_valid else float("nan")
    if reduction == "none":
        return loss_rows.copy()
    raise ValueError(f"reduction must be one of {REDUCTIONS}, got {reduction!r}")


def forward(hidden, weight, targets, bias=None, ignore_index: int = -100,
            logit_scale: float = 1.0, softcap: Optional[float] = None,
            z_loss_multiplier: float = 0.0, reduction: str = "mean",
            row_block: Optional[int] = None) -> dict:
    """Loss, per-row lse and metrics.

    ``row_block`` materialises the logits one block of rows at a time, to bound
    host memory. Every row is computed independently by the definition, so the
    result is the same as with all rows at once.
    """
    if reduction not in REDUCTIONS:
        raise ValueError(f"reduction must be one of {REDUCTIONS}, got {reduction!r}")
    targets = np.asarray(targets, dtype=np.int64)
    N = targets.shape[0]
    V = np.asarray(weight).shape[0]
    check_targets(targets, V, ignore_index)
    rb = row_block or max(N, 1)
    lse = np.empty(N)
    loss_rows = np.empty(N)
    entropy = np.empty(N)
    argmax = np.empty(N, dtype=np.int64)
    correct = np.zeros(N, dtype=bool)
    top2_gap = np.full(N, np.inf)
    valid = targets != ignore_index
    Wf = _f64(weight)
    bf = None if bias is None else _f64(bias)
    for r0 in range(0, N, rb):
        r1 = min(N, r0 + rb)
        z = transformed_logits(np.asarray(hidden)[r0:r1], Wf, bf, logit_scale, softcap)
        rt = row_terms(z, targets[r0:r1], ignore_index, z_loss_multiplier)
        lse[r0:r1] = rt["lse"]
        loss_rows[r0:r1] = rt["loss"]
        entropy[r0:r1] = rt["entropy"]
        argmax[r0:r1] = rt["argmax"]
        correct[r0:r1] = rt["correct"]
        if V > 1:
            top2 = np.partition(z, V - 2, axis=1)[:, V - 2:]
            top2_gap[r0:r1] = np.abs(top2[:, 1] - top2[:, 0])
    num_valid = int(valid.sum())
    return dict(
        loss=_reduce(loss_rows, num_valid, reduction),
        loss_rows=loss_rows,
        lse=lse,
        num_valid=num_valid,
        num_correct_tokens=int(correct.sum()),
        entropy_sum=float(entropy[valid].sum()),
        entropy_rows=entropy,
        argmax=argmax,
        correct=correct,
        top2_gap=top2_gap,
    )


def row_gamma(targets, ignore_index: int, reduction: str, grad_loss, num_valid: int) -> np.ndarray:
    """Upstream gradient of each row's loss term: d(reduced loss)/d(loss_i) times grad_loss."""
    t = np.asarray(targets, dtype=np.int64)
    valid = t != ignore_index
    if reduction == "none":
        g = _f64(grad_loss).reshape(-1)
        if g.shape[0] != t.shape[0]:
            raise ValueError("reduction='none' needs one grad_loss per row")
        gam = g.copy()
    elif reduction == "sum":
        gam = np.full(t.shape[0], float(np.asarray(grad_loss).reshape(-1)[0]))
    elif reduction == "mean":
        gl = float(np.asarray(grad_loss).reshape(-1)[0])
        gam = np.full(t.shape[0], gl / num_valid if num_valid else 0.0)
    else:
        raise ValueError(f"reduction must be one of {REDUCTIONS}, got {reduction!r}")
    return np.where(valid, gam, 0.0)


def dlogits(z: np.ndarray, lse: np.ndarray, targets, gamma: np.ndarray,
            logit_scale: float = 1.0, softcap: Optional[float] = None,
            z_loss_multiplier: float = 0.0) -> np.ndarray:
    """g = d(reduced loss) / d(a) for a block of rows, where a = h W^T is the raw projection.

    Chain rule through the loss terms, the softcap and the scale:
    dloss_i/dz_ij = p_ij (1 + 2 zeta lse_i) - [j == t_i]
    dz/du = 1 - (z/c)^2 (softcap only)
    du/da = s
    """
    t = np.asarray(targets, dtype=np.int64)
    n, V = z.shape
    p = np.exp(z - lse[:, None])
    g = p * (1.0 + 2.0 * float(z_loss_multiplier) * lse)[:, None]
    valid = gamma != 0.0
    rows = np.nonzero(valid & (t >= 0))[0]
    g[rows, t[rows]] -= 1.0
    if softcap is not None and softcap > 0:
        g = g * (1.0 - (z / float(softcap)) ** 2)
    g = g * (gamma * float(logit_scale))[:, None]
    g[~valid] = 0.0
    return g


def backward(hidden, weight, targets, bias=None, ignore_index: int = -100,
             logit_scale: float = 1.0, softcap: Optional[float] = None,
             z_loss_multiplier: float = 0.0, reduction: str = "mean",
             grad_loss=1.0, row_block: Optional[int] = None):
    """(grad_hidden [N,H], grad_weight [V,H], grad_bias [V] or None), all fp64."""
    targets = np.asarray(targets, dtype=np.int64)
    N = targets.shape[0]
    Wf = _f64(weight)
    V, H = Wf.shape
    check_targets(targets, V, ignore_index)
    num_valid = int((targets != ignore_index).sum())
    gamma = row_gamma(targets, ignore_index, reduction, grad_loss, num_valid)
    rb = row_block or max(N, 1)
    gh = np.zeros((N, H))
    gw = np.zeros((V, H))
    gb = np.zeros(V) if bias is not None else None
    hf_all = np.asarray(hidden)
    for r0 in range(0, N, rb):
        r1 = min(N, r0 + rb)
        hf = _f64(hf_all[r0:r1])
        z = transformed_logits(hf, Wf, bias, logit_scale, softcap)
        lse = row_terms(z, targets[r0:r1], ignore_index, z_loss_multiplier)["lse"]
        g = dlogits(z, lse, targets[r0:r1], gamma[r0:r1], logit_scale, softcap, z_loss_multiplier)
        gh[r0:r1] = g @ Wf
        gw += g.T @ hf
        if gb is not None:
            gb += g.sum(axis=0)
    return gh, gw, gb


# ---------------------------------------------------------------------------
# Sampled outputs, for full-size workloads. They compute, one output at a time,
# exactly the entries the functions above would produce.
# ---------------------------------------------------------------------------

def forward_rows(hidden, weight, targets, rows: Sequence[int], bias=None,
                 ignore_index: int = -100, logit_scale: float = 1.0,
                 softcap: Optional[float] = None, z_loss_multiplier: float = 0.0) -> dict:
    """lse, per-row loss, entropy, argmax and the top-2 logit gap, for the selected rows only."""
    rows = np.asarray(rows, dtype=np.int64)
    t = np.asarray(targets, dtype=np.int64)[rows]
    check_targets(t, np.asarray(weight).shape[0], ignore_index)
    z = transformed_logits(np.asarray(hidden)[rows], weight, bias, logit_scale, softcap)
    rt = row_terms(z, t, ignore_index, z_loss_multiplier)
    zs = np.sort(z, axis=1)
    gap = zs[:, -1] - zs[:, -2] if z.shape[1] > 1 else np.full(len(rows), np.inf)
    return dict(lse=rt["lse"], loss=rt["loss"], entropy=rt["entropy"], argmax=rt["argmax"],
                correct=rt["correct"], valid=rt["valid"], top2_gap=gap)


def grad_hidden_rows(hidden, weight, targets, rows: Sequence[int], bias=None,
                     ignore_index: int = -100, logit_scale: float = 1.0,
                     softcap: Optional[float] = None, z_loss_multiplier: float = 0.0,
                     reduction: str = "mean", grad_loss=1.0) -> np.ndarray:
    """grad_hidden[rows, :]. A row's gradient needs only that row's logits."""
    rows = np.asarray(rows, dtype=np.int64)
    tall = np.asarray(targets, dtype=np.int64)
    num_valid = int((tall != ignore_index).sum())
    gamma = row_gamma(tall, ignore_index, reduction, grad_loss, num_valid)[rows]
    Wf = _f64(weight)
    z = transformed_logits(np.asarray(hidden)[rows], Wf, bias, logit_scale, softcap)
    lse = row_terms(z, tall[rows], ignore_index, z_loss_multiplier)["lse"]
    g = dlogits(z, lse, tall[rows], gamma, logit_scale, softcap, z_loss_multiplier)
    return g @ Wf


def grad_weight_rows(hidden, weight, targets, lse_all: np.ndarray, vocab_rows: Sequence[int],
                     bias=None, ignore_index: int = -100, logit_scale: float = 1.0,
                     softcap: Optional[float] = None, z_loss_multiplier: float = 0.0,
                     reduction: str = "mean", grad_loss=1.0):
    """(grad_weight[vocab_rows, :], grad_bias[vocab_rows] or None).

    ``lse_all`` must be the oracle's own lse for every row, from ``forward``.
    A vocab row's gradient needs column j of the logits for all rows, plus each
    row's lse.
    """
    J = np.asarray(vocab_rows, dtype=np.int64)
    tall = np.asarray(targets, dtype=np.int64)
    N = tall.shape[0]
    num_valid = int((tall != ignore_index).sum())
    gamma = row_gamma(tall, ignore_index, reduction, grad_loss, num_valid)
    hf = _f64(hidden)
    zcols = transformed_logits(hf, _f64(weight)[J], None if bias is None else _f64(bias)[J],
                               logit_scale, softcap)  # [N, |J|]
    p = np.exp(zcols - lse_all[:, None])
    g = p * (1.0 + 2.0 * float(z_loss_multiplier) * lse_all)[:, None]
    onehot = (tall[:, None] == J[None, :])
    g = g - onehot
    if softcap is not None and softcap > 0:
        g = g * (1.0 - (zcols / float(softcap)) ** 2)
    g = g * (gamma * float(logit_scale))[:, None]
    g[gamma == 0.0] = 0.0
    gw = g.T @ hf
    gb = g.sum(axis=0) if bias is not None else None
    return gw, gb
