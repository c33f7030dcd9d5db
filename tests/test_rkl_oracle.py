"""Pins for the oracle's reverse KL over the cached ids: brute-force restated
definition on tiny inputs, torch autograd, finite differences, zero when the
student's restricted distribution equals the teacher's, and -inf teacher
entries leaving the support."""
import math

import numpy as np
import pytest
import torch

import oracle.kl_oracle as ok
from tests.test_oracle_pins import _rand_problem


def test_brute_force_small():
    rng = np.random.default_rng(0)
    H, W, idx, logit, mask = _rand_problem(rng, 3, 4, 9, 3, mask_p=1.0)
    tau = 1.5
    loss, rkl, _ = ok.reverse_kl_forward(H, W, idx, logit, mask, tau)
    for t in range(3):
        z = [float(H[t] @ W[v]) / tau for v in idx[t]]
        l = [x / tau for x in logit[t]]
        sz, sl = sum(math.exp(x) for x in z), sum(math.exp(x) for x in l)
        q = [math.exp(x) / sz for x in z]
        p = [math.exp(x) / sl for x in l]
        want = sum(qk * (math.log(qk) - math.log(pk)) for qk, pk in zip(q, p))
        assert abs(rkl[t] - want) < 1e-12
    assert abs(loss - rkl.mean()) < 1e-14


@pytest.mark.parametrize("tau", [1.0, 2.0])
def test_against_torch_autograd(tau):
    rng = np.random.default_rng(1)
    T, d, V, K = 6, 8, 30, 5
    H, W, idx, logit, mask = _rand_problem(rng, T, d, V, K)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    z = torch.gather(Ht @ Wt.T, 1, torch.tensor(idx)) / tau
    logq = torch.log_softmax(z, 1)
    logp = torch.log_softmax(torch.tensor(logit) / tau, 1)
    rkl = (logq.exp() * (logq - logp)).sum(1)
    m = torch.tensor(mask != 0, dtype=torch.float64)
    loss = (rkl * m).sum() / m.sum()
    (0.7 * loss).backward()
    o = ok.reverse_kl_forward(H, W, idx, logit, mask, tau)
    assert abs(o[0] - loss.item()) < 1e-12
    dH, dW = ok.reverse_kl_backward(H, W, idx, logit, mask, tau, 0.7)
    np.testing.assert_allclose(dH, Ht.grad.numpy(), rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-10, atol=1e-14)


def test_zero_when_distributions_match():
    rng = np.random.default_rng(2)
    H, W, idx, _, mask = _rand_problem(rng, 5, 6, 20, 4, mask_p=1.0)
    logit = np.take_along_axis(H @ W.T, idx, axis=1) + 3.0  # same up to a row constant
    loss, rkl, _ = ok.reverse_kl_forward(H, W, idx, logit, mask, 1.3)
    assert np.abs(rkl).max() < 1e-13
    dH, dW = ok.reverse_kl_backward(H, W, idx, logit, mask, 1.3)
    assert np.abs(dH).max() < 1e-13 and np.abs(dW).max() < 1e-13


def test_neg_inf_teacher_entry_leaves_the_support():
    rng = np.random.default_rng(3)
    H, W, idx, logit, mask = _rand_problem(rng, 4, 5, 15, 3, mask_p=1.0)
    extra = np.array([[v for v in range(15) if v not in row][0] for row in idx])
    idx2 = np.concatenate([idx, extra[:, None]], axis=1)
    logit2 = np.concatenate([logit, np.full((4, 1), -np.inf)], axis=1)
    a = ok.reverse_kl_forward(H, W, idx, logit, mask, 1.0)
    b = ok.reverse_kl_forward(H, W, idx2, logit2, mask, 1.0)
    assert abs(a[0] - b[0]) < 1e-13
    np.testing.assert_allclose(ok.reverse_kl_backward(H, W, idx, logit, mask, 1.0)[1],
                               ok.reverse_kl_backward(H, W, idx2, logit2, mask, 1.0)[1], atol=1e-15)


def test_finite_differences():
    rng = np.random.default_rng(4)
    H, W, idx, logit, mask = _rand_problem(rng, 3, 4, 7, 3)
    dH, dW = ok.reverse_kl_backward(H, W, idx, logit, mask, 2.0)
    h = 1e-6
    num = np.zeros_like(H)
    for i in range(H.shape[0]):
        for j in range(H.shape[1]):
            Hp, Hm = H.copy(), H.copy()
            Hp[i, j] += h
            Hm[i, j] -= h
            num[i, j] = (ok.reverse_kl_forward(Hp, W, idx, logit, mask, 2.0)[0] -
                         ok.reverse_kl_forward(Hm, W, idx, logit, mask, 2.0)[0]) / (2 * h)
    assert np.linalg.norm(dH - num) / np.linalg.norm(num) < 1e-7


@pytest.mark.parametrize("tau", [1.0, 0.5])
def test_grad_z_against_torch_autograd(tau):
    """dloss/dz at the cached ids, taken by autograd with the gathered logits
    as the leaf (masked tokens and -inf teacher entries included)."""
    rng = np.random.default_rng(7)
    T, d, V, K = 7, 6, 25, 6
    H, W, idx, logit, mask = _rand_problem(rng, T, d, V, K)
    logit[1, 2] = -np.inf
    z = torch.tensor(np.take_along_axis(H @ W.T, idx, axis=1), requires_grad=True)
    m = torch.tensor(mask != 0, dtype=torch.float64)
    rows = []
    for t in range(T):  # each row over its own support only
        keep = torch.tensor(np.flatnonzero(np.isfinite(logit[t])))
        logq = torch.log_softmax(z[t, keep] / tau, 0)
        logp = torch.log_softmax(torch.tensor(logit[t])[keep] / tau, 0)
        rows.append((logq.exp() * (logq - logp)).sum())
    loss = (torch.stack(rows) * m).sum() / m.sum()
    loss.backward()
    gz = ok.reverse_kl_grad_z(H, W, idx, logit, mask, tau)
    np.testing.assert_allclose(gz, z.grad.numpy(), rtol=1e-10, atol=1e-14)
    assert np.all(gz[mask == 0] == 0.0) and gz[1, 2] == 0.0
