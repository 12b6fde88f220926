"""Pins for the fp64 oracle. Each test checks it against something other than itself.

The pins are:
* torch's fp64 autograd through ``F.cross_entropy(F.linear(...))``. This is the
  library routine the quack reference names (quack-kernels diff,
  ``linear_cross_entropy_func_ref``). It covers loss and all three gradients
  when there is no softcap and no z-loss.
* central finite differences of the oracle's own loss, for the gradients with
  softcap and z-loss.
* closed forms: W = 0 gives ln V; V = 2 gives softplus; V = 1 gives 0; the
  hand-derived golden cases.
* invariants: shifting the bias, permuting the vocabulary, ignored rows,
  chunked sums ("Chunked Linear Loss", "Reduction semantics"), online merge over
  vocabulary splits (fused-linear-ce README, "Algorithm").
* brute force for the metrics (fused-linear-ce README, "Metrics for free").
* the row-sampled entry points (one row of grad_hidden, one vocabulary row of
  grad_weight, a few rows of the forward), which the full-size GPU tests use,
  against the full backward and forward, with softcap, z-loss, bias and
  ignored rows.

Each pin is chosen so that a plausible slip fails at least one of them: a
dropped term, a wrong sign, a transposed operand or a wrong reduction.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(seed, N, H, V, bias=True, ignore=(), scale=1.0):
    g = np.random.default_rng(seed)
    h = g.standard_normal((N, H))
    W = g.standard_normal((V, H)) * scale
    b = g.standard_normal(V) * 0.5 if bias else None
    t = g.integers(0, V, N)
    for i in ignore:
        t[i] = -100
    return h, W, b, t


def torch_ref(h, W, b, t, reduction, s=1.0, grad=None):
    ht = torch.tensor(h, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    bt = torch.tensor(b, dtype=torch.float64, requires_grad=True) if b is not None else None
    y = F.linear(ht, Wt, bt) * s
    loss = F.cross_entropy(y, torch.tensor(t), ignore_index=-100, reduction=reduction)
    if reduction == "none":
        loss.backward(torch.tensor(grad, dtype=torch.float64))
    else:
        loss.backward(torch.tensor(grad if grad is not None else 1.0, dtype=torch.float64))
    return (loss.detach().numpy(), ht.grad.numpy(), Wt.grad.numpy(),
            None if bt is None else bt.grad.numpy())


@pytest.mark.parametrize("reduction", ["sum", "mean", "none"])
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("scale", [1.0, 0.7, -1.3])
def test_matches_torch_cross_entropy(reduction, with_bias, scale):
    h, W, b, t = rnd(1, 9, 6, 13, bias=with_bias, ignore=(2, 5))
    g = np.random.default_rng(7).standard_normal(9) if reduction == "none" else 0.8
    ref_loss, ref_gh, ref_gw, ref_gb = torch_ref(h, W, b, t, reduction, scale, g)
    out = oracle.forward(h, W, t, bias=b, logit_scale=scale, reduction=reduction)
    gh, gw, gb = oracle.backward(h, W, t, bias=b, logit_scale=scale, reduction=reduction,
                                 grad_loss=g)
    np.testing.assert_allclose(out["loss"], ref_loss, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(gh, ref_gh, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(gw, ref_gw, rtol=1e-11, atol=1e-13)
    if with_bias:
        np.testing.assert_allclose(gb, ref_gb, rtol=1e-11, atol=1e-13)
    # the row-sampled entry points agree with the full ones
    rows = [0, 3, 8]
    np.testing.assert_allclose(
        oracle.grad_hidden_rows(h, W, t, rows, bias=b, logit_scale=scale, reduction=reduction,
                                grad_loss=g), gh[rows], rtol=1e-12, atol=1e-14)
    J = [0, 4, 12]
    gwJ, gbJ = oracle.grad_weight_rows(h, W, t, out["lse"], J, bias=b, logit_scale=scale,
                                       reduction=reduction, grad_loss=g)
    np.testing.assert_allclose(gwJ, gw[J], rtol=1e-12, atol=1e-14)
    if with_bias:
        np.testing.assert_allclose(gbJ, gb[J], rtol=1e-12, atol=1e-14)
    fr = oracle.forward_rows(h, W, t, rows, bias=b, logit_scale=scale)
    np.testing.assert_allclose(fr["loss"], out["loss_rows"][rows], rtol=1e-13)
    np.testing.assert_allclose(fr["lse"], out["lse"][rows], rtol=1e-13)


@pytest.mark.parametrize("reduction", ["sum", "mean", "none"])
@pytest.mark.parametrize("softcap,zeta,scale", [(None, 0.3, 1.0), (2.0, 0.0, 0.6),
                                                (1.5, 0.2, -0.8)])
def test_row_sampled_entry_points_with_softcap_and_zloss(reduction, softcap, zeta, scale):
    """The sampled entry points the full-size GPU tests use (one row of
    grad_hidden, one vocabulary row of grad_weight / grad_bias, the forward of
    a few rows) agree with the full backward and forward, which the finite
    differences and torch autograd pin, with the softcap and z-loss factors,
    ignored rows and a bias."""
    h, W, b, t = rnd(5, 10, 6, 11, bias=True, ignore=(1, 6))
    g = np.random.default_rng(9).standard_normal(10) if reduction == "none" else 1.3
    kw = dict(bias=b, logit_scale=scale, softcap=softcap, z_loss_multiplier=zeta)
    out = oracle.forward(h, W, t, reduction=reduction, **kw)
    gh, gw, gb = oracle.backward(h, W, t, reduction=reduction, grad_loss=g, **kw)
    rows = [0, 1, 4, 9]
    np.testing.assert_allclose(
        oracle.grad_hidden_rows(h, W, t, rows, reduction=reduction, grad_loss=g, **kw),
        gh[rows], rtol=1e-12, atol=1e-14)
    J = [0, 3, 10]
    gwJ, gbJ = oracle.grad_weight_rows(h, W, t, out["lse"], J, reduction=reduction,
                                       grad_loss=g, **kw)
    np.testing.assert_allclose(gwJ, gw[J], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(gbJ, gb[J], rtol=1e-12, atol=1e-14)
    fr = oracle.forward_rows(h, W, t, rows, **kw)
    np.testing.assert_allclose(fr["loss"], out["loss_rows"][rows], rtol=1e-13)
    np.testing.assert_allclose(fr["lse"], out["lse"][rows], rtol=1e-13)
    np.testing.assert_allclose(fr["entropy"], out["entropy_rows"][rows], rtol=1e-12)


def test_lse_matches_torch_logsumexp():
    h, W, b, t = rnd(2, 5, 4, 30)
    out = oracle.forward(h, W, t, bias=b, logit_scale=2.5)
    y = torch.tensor((h @ W.T + b) * 2.5)
    np.testing.assert_allclose(out["lse"], torch.logsumexp(y, dim=1).numpy(), rtol=1e-14)


def _loss_for_fd(h, W, b, t, kw, weights):
    out = oracle.forward(h, W, t, bias=b, **kw)
    if kw["reduction"] == "none":
        return float(np.dot(out["loss"], weights))
    return out["loss"]


@pytest.mark.parametrize("reduction", ["sum", "mean", "none"])
@pytest.mark.parametrize("softcap,zeta,scale", [(None, 0.3, 1.0), (2.0, 0.0, 0.6),
                                                (1.5, 0.2, -0.8)])
def test_finite_differences(reduction, softcap, zeta, scale):
    """Central differences of the oracle loss agree with its analytic gradients, including softcap and z-loss."""
    h, W, b, t = rnd(3, 4, 3, 6, ignore=(1,))
    weights = np.array([0.3, -1.2, 0.9, 2.0])
    kw = dict(logit_scale=scale, softcap=softcap, z_loss_multiplier=zeta, reduction=reduction)
    gl = weights if reduction == "none" else 1.0
    gh, gw, gb = oracle.backward(h, W, t, bias=b, grad_loss=gl, **kw)
    eps = 1e-6
    for arr, grad in ((h, gh), (W, gw), (b, gb)):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + eps
            lp = _loss_for_fd(h, W, b, t, kw, weights)
            arr[idx] = old - eps
            lm = _loss_for_fd(h, W, b, t, kw, weights)
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8)


def test_autograd_of_softcap_and_zloss_gradients():
    """torch autograd through an independent graph of the loss with tanh softcap and z-loss.

    The graph uses torch.logsumexp and gather. It checks the oracle's
    hand-derived chain rule.
    """
    h, W, b, t = rnd(4, 6, 5, 9, ignore=(0,))
    s, c, zeta = 0.9, 3.0, 0.05
    ht = torch.tensor(h, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    bt = torch.tensor(b, requires_grad=True)
    z = c * torch.tanh(F.linear(ht, Wt, bt) * s / c)
    lse = torch.logsumexp(z, dim=1)
    tt = torch.tensor(t)
    valid = tt != -100
    zt = z.gather(1, tt.clamp(min=0)[:, None])[:, 0]
    loss = torch.where(valid, lse - zt + zeta * lse ** 2, torch.zeros_like(lse)).sum() / valid.sum()
    loss.backward()
    out = oracle.forward(h, W, t, bias=b, logit_scale=s, softcap=c, z_loss_multiplier=zeta,
                         reduction="mean")
    gh, gw, gb = oracle.backward(h, W, t, bias=b, logit_scale=s, softcap=c,
                                 z_loss_multiplier=zeta, reduction="mean")
    np.testing.assert_allclose(out["loss"], loss.item(), rtol=1e-13)
    np.testing.assert_allclose(gh, ht.grad.numpy(), rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(gw, Wt.grad.numpy(), rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(gb, bt.grad.numpy(), rtol=1e-11, atol=1e-14)


def test_huge_softcap_reduces_to_plain_cross_entropy():
    h, W, b, t = rnd(5, 5, 4, 7)
    ref = torch_ref(h, W, b, t, "mean")
    out = oracle.forward(h, W, t, bias=b, softcap=1e7, reduction="mean")
    gh, gw, gb = oracle.backward(h, W, t, bias=b, softcap=1e7, reduction="mean")
    np.testing.assert_allclose(out["loss"], ref[0], rtol=1e-9)
    np.testing.assert_allclose(gw, ref[2], rtol=1e-8, atol=1e-12)


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "hand_cases.json")))["cases"],
                         ids=lambda c: c["name"])
def test_golden_hand_cases(case):
    kw = dict(logit_scale=case["logit_scale"], softcap=case["softcap"],
              z_loss_multiplier=case["z_loss_multiplier"], reduction=case["reduction"])
    h = np.array(case["hidden"])
    W = np.array(case["weight"])
    b = None if case["bias"] is None else np.array(case["bias"])
    t = np.array(case["targets"])
    e = case["expect"]
    out = oracle.forward(h, W, t, bias=b, **kw)
    gh, gw, gb = oracle.backward(h, W, t, bias=b, grad_loss=case["grad_loss"], **kw)
    assert out["loss"] == pytest.approx(e["loss"], rel=1e-13)
    np.testing.assert_allclose(out["lse"], e["lse"], rtol=1e-13)
    assert out["entropy_sum"] == pytest.approx(e["entropy_sum"], rel=1e-13)
    assert out["num_correct_tokens"] == e["num_correct_tokens"]
    np.testing.assert_allclose(gh, e["grad_hidden"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(gw, e["grad_weight"], rtol=1e-12, atol=1e-15)
    if e["grad_bias"] is not None:
        np.testing.assert_allclose(gb, e["grad_bias"], rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("zeta", [0.0, 1e-4, 0.5])
def test_zero_weight_gives_log_v(zeta):
    V = 37
    h = np.random.default_rng(0).standard_normal((6, 5))
    W = np.zeros((V, 5))
    t = np.array([0, 36, -100, 5, 5, 17])
    out = oracle.forward(h, W, t, bias=np.zeros(V), z_loss_multiplier=zeta, reduction="none")
    lv = math.log(V)
    expect = np.where(t != -100, lv + zeta * lv * lv, 0.0)
    np.testing.assert_allclose(out["loss"], expect, rtol=1e-14)
    np.testing.assert_allclose(out["entropy_rows"], lv, rtol=1e-14)
    assert (out["argmax"] == 0).all()  # every logit ties; the lowest index wins
    assert out["num_correct_tokens"] == 1  # only the row with target 0


def test_two_classes_softplus_and_one_class_zero():
    h, W, b, t = rnd(6, 8, 3, 2)
    z = h @ W.T + b
    out = oracle.forward(h, W, t, bias=b, reduction="none")
    other = z[np.arange(8), 1 - t]
    mine = z[np.arange(8), t]
    np.testing.assert_allclose(out["loss"], np.logaddexp(0.0, other - mine), rtol=1e-13)
    h1, W1, b1, _ = rnd(7, 4, 3, 1)
    out1 = oracle.forward(h1, W1, np.zeros(4, dtype=np.int64), bias=b1, reduction="sum")
    assert out1["loss"] == 0.0 and out1["entropy_sum"] == 0.0
    gh, gw, gb = oracle.backward(h1, W1, np.zeros(4, dtype=np.int64), bias=b1, reduction="sum")
    assert np.abs(gh).max() == 0 and np.abs(gw).max() == 0 and np.abs(gb).max() == 0


@pytest.mark.parametrize("shift", [3.25, 1000.0])
def test_bias_shift_invariance(shift):
    """A constant added to every logit changes nothing. At a shift of 1000 the
    logits are far past exp's fp64 overflow (about 709), so this also pins the
    max subtraction; the shift cancels in fp64 to about shift x 2^-52."""
    h, W, b, t = rnd(8, 7, 4, 11, ignore=(3,))
    a = oracle.forward(h, W, t, bias=b, reduction="mean", logit_scale=1.7)
    c = oracle.forward(h, W, t, bias=b + shift / 1.7, reduction="mean", logit_scale=1.7)
    assert np.isfinite(c["loss"])
    assert a["loss"] == pytest.approx(c["loss"], rel=1e-12)
    ga = oracle.backward(h, W, t, bias=b, reduction="mean", logit_scale=1.7)
    gc = oracle.backward(h, W, t, bias=b + shift / 1.7, reduction="mean", logit_scale=1.7)
    for x, y in zip(ga, gc):
        np.testing.assert_allclose(x, y, rtol=1e-10, atol=1e-13)


def test_vocab_permutation_invariance():
    h, W, b, t = rnd(9, 6, 4, 10, ignore=(4,))
    perm = np.random.default_rng(1).permutation(10)
    inv = np.argsort(perm)
    t2 = np.where(t >= 0, inv[np.maximum(t, 0)], t)
    kw = dict(softcap=2.0, z_loss_multiplier=0.01, reduction="sum", logit_scale=1.2)
    a = oracle.forward(h, W, t, bias=b, **kw)
    c = oracle.forward(h, W[perm], t2, bias=b[perm], **kw)
    assert a["loss"] == pytest.approx(c["loss"], rel=1e-13)
    assert a["entropy_sum"] == pytest.approx(c["entropy_sum"], rel=1e-13)
    ga = oracle.backward(h, W, t, bias=b, **kw)
    gc = oracle.backward(h, W[perm], t2, bias=b[perm], **kw)
    np.testing.assert_allclose(ga[0], gc[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ga[1][perm], gc[1], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ga[2][perm], gc[2], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("zeta", [0.0, 0.25])
def test_dlogit_row_sums(zeta):
    """Before the gamma, softcap and scale factors, a valid row of dloss/dz sums to 0, or to 2 zeta lse with z-loss."""
    h, W, b, t = rnd(10, 5, 4, 9, ignore=(2,))
    z = oracle.transformed_logits(h, W, b)
    lse = oracle.row_terms(z, t, -100)["lse"]
    gamma = np.where(t != -100, 1.0, 0.0)
    g = oracle.dlogits(z, lse, t, gamma, z_loss_multiplier=zeta)
    sums = g.sum(axis=1)
    np.testing.assert_allclose(sums[t != -100], (2 * zeta * lse)[t != -100], atol=1e-13)
    assert np.abs(g[2]).max() == 0.0


def test_ignored_rows_contribute_nothing():
    h, W, b, t = rnd(11, 8, 4, 9, ignore=(1, 6))
    kw = dict(softcap=4.0, z_loss_multiplier=0.1, reduction="sum")
    out = oracle.forward(h, W, t, bias=b, **{**kw, "reduction": "none"})
    assert out["loss"][1] == 0.0 and out["loss"][6] == 0.0
    gh, gw, gb = oracle.backward(h, W, t, bias=b, **kw)
    assert np.abs(gh[[1, 6]]).max() == 0.0
    keep = [0, 2, 3, 4, 5, 7]
    gh2, gw2, gb2 = oracle.backward(h[keep], W, t[keep], bias=b, **kw)
    np.testing.assert_allclose(gw, gw2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(gb, gb2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(gh[keep], gh2, rtol=1e-13, atol=1e-15)


def test_chunked_sum_equals_full_and_chunk_means_do_not():
    """'Chunked Linear Loss', 'Reduction semantics': chunk sums add up; a mean needs the global valid count."""
    h, W, b, t = rnd(12, 12, 4, 9, ignore=(0, 1, 2, 9))  # chunk masks differ
    full = oracle.forward(h, W, t, bias=b, reduction="sum")
    gfull = oracle.backward(h, W, t, bias=b, reduction="sum")
    chunks = [(0, 4), (4, 7), (7, 12)]
    s = 0.0
    gw = np.zeros_like(W)
    cnt = 0
    chunk_means = []
    for r0, r1 in chunks:
        o = oracle.forward(h[r0:r1], W, t[r0:r1], bias=b, reduction="sum")
        s += o["loss"]
        cnt += o["num_valid"]
        chunk_means.append(oracle.forward(h[r0:r1], W, t[r0:r1], bias=b, reduction="mean")["loss"])
        gw += oracle.backward(h[r0:r1], W, t[r0:r1], bias=b, reduction="sum")[1]
    assert s == pytest.approx(full["loss"], rel=1e-13)
    np.testing.assert_allclose(gw, gfull[1], rtol=1e-12, atol=1e-14)
    mean = oracle.forward(h, W, t, bias=b, reduction="mean")["loss"]
    assert mean == pytest.approx(s / cnt, rel=1e-13)
    assert abs(np.mean(chunk_means) - mean) > 1e-3


def _partial_state(z_block, col0):
    """Running (max, sum exp, sum z exp, argmax) over one block of columns, as a vocabulary-tiled pass keeps it."""
    m = z_block.max(axis=1)
    e = np.exp(z_block - m[:, None])
    return m, e.sum(axis=1), (z_block * e).sum(axis=1), col0 + z_block.argmax(axis=1)


def test_vocab_split_online_merge_equals_full_row():
    """fused-linear-ce README, "Algorithm": merging vocabulary tiles with online-softmax rescaling.

    The merged state must give the oracle's lse, entropy and argmax. The
    splits are uneven and the last one is ragged.
    """
    h, W, b, t = rnd(13, 6, 5, 50)
    z = oracle.transformed_logits(h, W, b, softcap=3.0)
    ref = oracle.forward(h, W, t, bias=b, softcap=3.0, reduction="none")
    bounds = [0, 7, 8, 31, 50]
    m = np.full(6, -np.inf)
    s = np.zeros(6)
    tt = np.zeros(6)
    am = np.zeros(6, dtype=np.int64)
    for c0, c1 in zip(bounds[:-1], bounds[1:]):
        mk, sk, tk, ak = _partial_state(z[:, c0:c1], c0)
        mn = np.maximum(m, mk)
        am = np.where(mk > m, ak, am)
        s = s * np.exp(m - mn) + sk * np.exp(mk - mn)
        tt = tt * np.exp(m - mn) + tk * np.exp(mk - mn)
        m = mn
    lse = m + np.log(s)
    np.testing.assert_allclose(lse, ref["lse"], rtol=1e-14)
    np.testing.assert_allclose(lse - tt / s, ref["entropy_rows"], rtol=1e-12)
    np.testing.assert_array_equal(am, ref["argmax"])


def test_metrics_brute_force():
    h, W, b, t = rnd(14, 10, 3, 7, ignore=(3,))
    W[2] = W[5]  # make exact ties in the argmax
    b[2] = b[5]
    t[0] = 2
    out = oracle.forward(h, W, t, bias=b, reduction="sum")
    z = (h @ W.T + b).tolist()
    correct = 0
    ent = 0.0
    for i, row in enumerate(z):
        best = 0
        for j in range(len(row)):
            if row[j] > row[best]:
                best = j
        assert out["argmax"][i] == best
        if t[i] == -100:
            continue
        correct += int(best == t[i])
        mx = max(row)
        den = sum(math.exp(v - mx) for v in row)
        ent -= sum((math.exp(v - mx) / den) * math.log(math.exp(v - mx) / den) for v in row)
    assert out["num_correct_tokens"] == correct
    assert out["entropy_sum"] == pytest.approx(ent, rel=1e-12)


def brute_top2_gap(row):
    """Largest value minus the second largest of a list, by one scan (ties give 0)."""
    if len(row) < 2:
        return math.inf
    best, second = -math.inf, -math.inf
    for v in row:
        if v > best:
            best, second = v, best
        elif v > second:
            second = v
    return best - second


def plain_logits(h, W, b, s=1.0, c=None):
    """z_ij written out element by element (bias, then scale, then the tanh softcap)."""
    z = []
    for hi in h.tolist():
        row = []
        for j, wj in enumerate(W.tolist()):
            u = (sum(x * y for x, y in zip(hi, wj)) + (0.0 if b is None else float(b[j]))) * s
            row.append(c * math.tanh(u / c) if c else u)
        z.append(row)
    return z


@pytest.mark.parametrize("V", [1, 2, 3, 9])
def test_top2_gap_brute_force(V):
    """top2_gap, which excuses near-tie rows from the exact num_correct check, is the
    largest logit minus the second largest, in both forward and forward_rows."""
    h, W, b, t = rnd(40 + V, 12, 4, V)
    if V >= 3:
        W[0] *= 2.0          # column 0 leads in many rows ...
        b[0] = 2.0
        W[2] = W[0]          # ... tied with column 2: gap 0 there
        b[2] = b[0]
    kw = dict(logit_scale=0.8, softcap=3.0)
    z = plain_logits(h, W, b, s=0.8, c=3.0)
    want = np.array([brute_top2_gap(row) for row in z])
    out = oracle.forward(h, W, t, bias=b, reduction="none", **kw)
    blk = oracle.forward(h, W, t, bias=b, reduction="none", row_block=5, **kw)
    rows = [0, 3, 7, 11]
    fr = oracle.forward_rows(h, W, t, rows, bias=b, **kw)
    if V == 1:
        assert np.isinf(out["top2_gap"]).all() and np.isinf(fr["top2_gap"]).all()
        return
    np.testing.assert_allclose(out["top2_gap"], want, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(blk["top2_gap"], want, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fr["top2_gap"], want[rows], rtol=1e-12, atol=1e-13)
    assert (out["top2_gap"] >= 0).all()
    if V >= 3:
        # rows whose top logit is the tied pair (columns 0 and 2) have gap 0
        tied = [i for i, row in enumerate(z) if max(row) == row[0]]
        assert tied and all(out["top2_gap"][i] == 0.0 for i in tied)


def test_mean_with_every_row_ignored():
    h, W, b, t = rnd(16, 4, 3, 5, ignore=(0, 1, 2, 3))
    out = oracle.forward(h, W, t, bias=b, reduction="mean")
    ref = torch_ref(h, W, None, t, "mean")
    assert math.isnan(out["loss"]) and math.isnan(float(ref[0]))
    gh, gw, gb = oracle.backward(h, W, t, bias=b, reduction="mean")
    assert not np.abs(gh).any() and not np.abs(gw).any() and not np.abs(gb).any()


def test_out_of_range_target_is_an_error():
    h, W, b, t = rnd(17, 3, 2, 4)
    t[1] = 4
    with pytest.raises(ValueError):
        oracle.forward(h, W, t)
    t[1] = -5
    with pytest.raises(ValueError):
        oracle.backward(h, W, t)


def test_row_block_gives_identical_result():
    h, W, b, t = rnd(18, 11, 4, 9, ignore=(5,))
    a = oracle.forward(h, W, t, bias=b, reduction="none", softcap=2.0)
    c = oracle.forward(h, W, t, bias=b, reduction="none", softcap=2.0, row_block=3)
    np.testing.assert_array_equal(a["loss"], c["loss"])
    ga = oracle.backward(h, W, t, bias=b, softcap=2.0)
    gc = oracle.backward(h, W, t, bias=b, softcap=2.0, row_block=4)
    for x, y in zip(ga, gc):
        np.testing.assert_allclose(x, y, rtol=1e-13, atol=1e-15)
