"""Pins of the generic chunked-linear-loss oracle ("Chunked Linear Loss").

Each pin checks the oracle against something other than itself:
- torch fp64 autograd through F.linear and an independently written loss;
- central finite differences of the chunked loss;
- independence from the chunk size, which the page's additive-loss argument
  ("Why chunk the projection?") promises;
- the closed form at W = 0;
- the cross-entropy oracle of the fused path, on the same inputs.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def rnd(N=11, H=6, V=9, seed=0):
    g = np.random.default_rng(seed)
    X = g.standard_normal((N, H))
    W = g.standard_normal((V, H)) / np.sqrt(H)
    Y = g.standard_normal((N, V))
    r = g.uniform(0.2, 2.0, N)
    f = g.uniform(0.2, 2.0, V)
    return X, W, Y, r, f


def test_weighted_mse_matches_torch_autograd():
    X, W, Y, r, f = rnd()
    loss, dX, dW = oracle.chunked_linear_loss(X, W, oracle.weighted_mse, Y, r, f, chunk_rows=4)
    Xt = torch.tensor(X, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    z = F.linear(Xt, Wt)
    ref = (torch.tensor(r)[:, None] * torch.tensor(f)[None, :] * (z - torch.tensor(Y)) ** 2).sum()
    ref.backward()
    assert loss == pytest.approx(ref.item(), rel=1e-13)
    np.testing.assert_allclose(dX, Xt.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-12, atol=1e-13)


def test_cross_entropy_matches_torch_autograd_and_the_fused_oracle():
    X, W, _, _, _ = rnd(N=13, V=7, seed=3)
    t = np.random.default_rng(4).integers(0, 7, 13)
    t[[2, 9]] = -100
    loss, dX, dW = oracle.chunked_linear_loss(X, W, oracle.cross_entropy_sum, t, chunk_rows=5)
    Xt = torch.tensor(X, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    ref = F.cross_entropy(F.linear(Xt, Wt), torch.tensor(t), ignore_index=-100, reduction="sum")
    ref.backward()
    assert loss == pytest.approx(ref.item(), rel=1e-13)
    np.testing.assert_allclose(dX, Xt.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-12, atol=1e-13)
    fused = oracle.forward(X, W, t, reduction="sum")
    gh, gw, _ = oracle.backward(X, W, t, reduction="sum")
    assert loss == pytest.approx(fused["loss"], rel=1e-13)
    np.testing.assert_allclose(dX, gh, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dW, gw, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("which", ["X", "W"])
def test_finite_differences(which):
    X, W, Y, r, f = rnd(N=7, H=5, V=6, seed=7)
    _, dX, dW = oracle.chunked_linear_loss(X, W, oracle.weighted_mse, Y, r, f, chunk_rows=3)
    eps = 1e-6
    A, G = (X, dX) if which == "X" else (W, dW)
    g = np.random.default_rng(8)
    for _ in range(6):
        i, j = g.integers(0, A.shape[0]), g.integers(0, A.shape[1])
        Ap, Am = A.copy(), A.copy()
        Ap[i, j] += eps
        Am[i, j] -= eps
        args = (Ap, W) if which == "X" else (X, Ap)
        lp = oracle.chunked_linear_loss(*args, oracle.weighted_mse, Y, r, f, chunk_rows=3)[0]
        args = (Am, W) if which == "X" else (X, Am)
        lm = oracle.chunked_linear_loss(*args, oracle.weighted_mse, Y, r, f, chunk_rows=3)[0]
        assert (lp - lm) / (2 * eps) == pytest.approx(G[i, j], rel=1e-6, abs=1e-8)


def test_result_does_not_depend_on_the_chunk_size():
    X, W, Y, r, f = rnd(N=17, seed=11)
    ref = oracle.chunked_linear_loss(X, W, oracle.weighted_mse, Y, r, f, chunk_rows=17)
    for rows in (1, 2, 5, 16, 40):
        got = oracle.chunked_linear_loss(X, W, oracle.weighted_mse, Y, r, f, chunk_rows=rows)
        assert got[0] == pytest.approx(ref[0], rel=1e-13)
        np.testing.assert_allclose(got[1], ref[1], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(got[2], ref[2], rtol=1e-12, atol=1e-13)


def test_zero_weight_closed_form():
    """W = 0 gives z = 0: L = sum r f y^2, dX = 0, dW_jk = -2 f_j sum_i r_i y_ij X_ik."""
    X, W, Y, r, f = rnd(N=5, H=3, V=4, seed=13)
    W = np.zeros_like(W)
    loss, dX, dW = oracle.chunked_linear_loss(X, W, oracle.weighted_mse, Y, r, f, chunk_rows=2)
    expect_loss = sum(r[i] * f[j] * Y[i, j] ** 2 for i in range(5) for j in range(4))
    assert loss == pytest.approx(expect_loss, rel=1e-13)
    assert not dX.any()
    for j in range(4):
        for k in range(3):
            e = -2 * f[j] * sum(r[i] * Y[i, j] * X[i, k] for i in range(5))
            assert dW[j, k] == pytest.approx(e, rel=1e-12, abs=1e-14)


def test_sliced_and_passed_through_arguments():
    """Per-row arrays are sliced to the chunk; other values pass unchanged ("Sliced arguments")."""
    X, W, Y, r, f = rnd(N=6, V=9, seed=17)   # f has V = 9 entries, not one per row
    seen = []

    def fn(z, y, rw, fw, scale=1.0):
        seen.append((z.shape[0], y.shape[0], rw.shape[0], fw.shape[0], scale))
        loss, g = oracle.weighted_mse(z, y, rw, fw)
        return loss * scale, g * scale

    got = oracle.chunked_linear_loss(X, W, fn, Y, r, f, chunk_rows=4, scale=2.0)
    assert seen == [(4, 4, 4, 9, 2.0), (2, 2, 2, 9, 2.0)]
    ref = oracle.chunked_linear_loss(X, W, oracle.weighted_mse, Y, r, f)
    assert got[0] == pytest.approx(2 * ref[0], rel=1e-13)


def test_cross_entropy_is_shift_invariant_past_exp_overflow():
    """Adding 1000 to every logit (past exp's fp64 overflow near 709) changes
    neither the summed cross-entropy nor its gradient: the log-sum-exp must
    subtract the row maximum."""
    g = np.random.default_rng(17)
    z = g.standard_normal((9, 13))
    t = g.integers(0, 13, 9)
    t[2] = -100
    l0, g0 = oracle.cross_entropy_sum(z, t)
    l1, g1 = oracle.cross_entropy_sum(z + 1000.0, t)
    assert np.isfinite(l1)
    assert l1 == pytest.approx(l0, rel=1e-11)
    np.testing.assert_allclose(g1, g0, rtol=1e-9, atol=1e-12)
