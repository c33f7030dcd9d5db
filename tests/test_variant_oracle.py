"""Pins for the oracle's loss variant (alpha-weighted KL plus hard-label CE,
optional tau^2): special cases that reduce to the pinned KL oracle and to
torch's cross_entropy, torch autograd of the same mix, finite differences."""
import numpy as np
import pytest
import torch

import oracle.kl_oracle as ok
from tests.test_oracle_pins import _rand_problem


def _labels(rng, T, V):
    return rng.integers(0, V, size=T)


@pytest.mark.parametrize("tau", [1.0, 2.0])
def test_alpha_one_is_the_kl_loss(tau):
    rng = np.random.default_rng(1)
    H, W, idx, logit, mask = _rand_problem(rng, 9, 8, 30, 5)
    y = _labels(rng, 9, 30)
    a = ok.forward(H, W, idx, logit, mask, tau)
    b = ok.forward_mixed(H, W, idx, logit, mask, tau, 1.0, False, y)
    assert abs(a[0] - b[0]) < 1e-13
    np.testing.assert_allclose(ok.backward(H, W, idx, logit, mask, tau)[1],
                               ok.backward_mixed(H, W, idx, logit, mask, tau, 1.0, False, y)[1],
                               atol=1e-15)
    c = ok.forward_mixed(H, W, idx, logit, mask, tau, 1.0, True, y)
    assert abs(c[0] - tau * tau * a[0]) < 1e-12


def test_alpha_zero_is_cross_entropy():
    rng = np.random.default_rng(2)
    H, W, idx, logit, mask = _rand_problem(rng, 11, 6, 25, 4, mask_p=1.0)
    y = _labels(rng, 11, 25)
    loss, _, lse1, tok = ok.forward_mixed(H, W, idx, logit, mask, 2.0, 0.0, True, y)
    ce = torch.nn.functional.cross_entropy(torch.tensor(H @ W.T), torch.tensor(y), reduction="none")
    np.testing.assert_allclose(tok, ce.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse1, torch.logsumexp(torch.tensor(H @ W.T), 1).numpy(), rtol=1e-13)


@pytest.mark.parametrize("tau,alpha,sq", [(1.0, 0.3, False), (2.0, 0.6, True), (0.5, 0.9, True)])
def test_against_torch_autograd(tau, alpha, sq):
    rng = np.random.default_rng(3)
    T, d, V, K = 7, 10, 35, 6
    H, W, idx, logit, mask = _rand_problem(rng, T, d, V, K)
    y = _labels(rng, T, V)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    z = Ht @ Wt.T
    p = torch.softmax(torch.tensor(logit) / tau, 1)
    P = torch.zeros(T, V, dtype=torch.float64).scatter_add_(1, torch.tensor(idx), p)
    kl = torch.nn.functional.kl_div(torch.log_softmax(z / tau, 1), P, reduction="none").sum(1)
    ce = torch.nn.functional.cross_entropy(z, torch.tensor(y), reduction="none")
    m = torch.tensor(mask != 0, dtype=torch.float64)
    c = tau * tau if sq else 1.0
    loss = ((alpha * c * kl + (1 - alpha) * ce) * m).sum() / m.sum()
    (1.3 * loss).backward()
    o = ok.forward_mixed(H, W, idx, logit, mask, tau, alpha, sq, y)
    assert abs(o[0] - loss.item()) < 1e-12
    dH, dW = ok.backward_mixed(H, W, idx, logit, mask, tau, alpha, sq, y, 1.3)
    np.testing.assert_allclose(dH, Ht.grad.numpy(), rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-10, atol=1e-14)


def test_finite_differences_mixed():
    rng = np.random.default_rng(4)
    T, d, V, K, tau, alpha = 3, 4, 7, 3, 2.0, 0.4
    H, W, idx, logit, mask = _rand_problem(rng, T, d, V, K)
    y = _labels(rng, T, V)
    dH, dW = ok.backward_mixed(H, W, idx, logit, mask, tau, alpha, True, y)
    h = 1e-6
    num = np.zeros_like(W)
    for i in range(V):
        for j in range(d):
            Wp, Wm = W.copy(), W.copy()
            Wp[i, j] += h
            Wm[i, j] -= h
            num[i, j] = (ok.forward_mixed(H, Wp, idx, logit, mask, tau, alpha, True, y)[0] -
                         ok.forward_mixed(H, Wm, idx, logit, mask, tau, alpha, True, y)[0]) / (2 * h)
    assert np.linalg.norm(dW - num) / np.linalg.norm(num) < 1e-7
