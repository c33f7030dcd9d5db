"""Pins for the fp64 oracle: checks against what the mathematics fixes, none of
which re-types the oracle's own formulas.

* closed forms worked by hand (tests/golden/closed_form_cases.json);
* central finite differences of the oracle's own loss against its closed-form
  gradient (the pages name a closed-form gradient but never print it);
* torch autograd through library routines (log_softmax, kl_div, cross_entropy)
  in fp64 as an independent derivation;
* invariants: KL >= 0, KL = 0 when the teacher equals the student with K = V,
  shift invariance, permutation invariance over k, mask invariance,
  sum_v G = 0, dense-grid KL = gathered KL (the pages state the dense, chunked
  and fused variants are mathematically equivalent);
* planted mistakes: each plausible bug in a copy of the oracle fails a pin.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.kl_oracle as ok

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")
_SAFE = {"__builtins__": {}, "log": math.log, "sqrt": math.sqrt}


def _ev(x):
    return None if x is None else float(eval(str(x), _SAFE, {}))


def _evm(a):
    return np.array([[_ev(x) for x in row] for row in a], dtype=np.float64)


def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _rand_problem(rng, T, d, V, K, mask_p=0.7, distinct=True):
    H = rng.standard_normal((T, d))
    W = rng.standard_normal((V, d)) / math.sqrt(d)
    if distinct:
        idx = np.stack([rng.permutation(V)[:K] for _ in range(T)])
    else:
        idx = rng.integers(0, V, size=(T, K))
    logit = rng.standard_normal((T, K)) * 2.0
    mask = (rng.random(T) < mask_p).astype(np.uint8)
    if mask.sum() == 0:
        mask[0] = 1
    return H, W, idx, logit, mask


# ----------------------------------------------------------------- closed forms

@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_closed_form_cases(case):
    tau, g = _ev(case["tau"]), _ev(case["grad_loss"])
    H, W = _evm(case["H"]), _evm(case["W"])
    idx = np.array(case["topk_idx"], dtype=np.int64)
    logit = _evm(case["topk_logit"])
    mask = np.array(case["mask"], dtype=np.uint8)
    ex = case["expect"]
    loss, lse, kl = ok.forward(H, W, idx, logit, mask, tau)
    assert abs(loss - _ev(ex["loss"])) < 1e-14
    for t, (e_lse, e_kl) in enumerate(zip(ex["lse"], ex["token_kl"])):
        if e_lse is not None:
            assert abs(lse[t] - _ev(e_lse)) < 1e-14
            assert abs(kl[t] - _ev(e_kl)) < 1e-14
    dH, dW = ok.backward(H, W, idx, logit, mask, tau, g)
    np.testing.assert_allclose(dH, _evm(ex["dH"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dW, _evm(ex["dW"]), rtol=0, atol=1e-14)


# ----------------------------------------------------------- finite differences

@pytest.mark.parametrize("K", [1, 3, 7])
@pytest.mark.parametrize("tau", [1.0, 2.0])
def test_finite_differences(K, tau):
    rng = np.random.default_rng(100 + 10 * K + int(tau))
    T, d, V = 3, 4, 7
    H, W, idx, logit, mask = _rand_problem(rng, T, d, V, K)
    g = 1.7
    dH, dW = ok.backward(H, W, idx, logit, mask, tau, g)

    def L(Hx, Wx):
        return g * ok.forward(Hx, Wx, idx, logit, mask, tau)[0]

    h = 1e-6
    num_dH = np.zeros_like(H)
    for i in range(T):
        for j in range(d):
            Hp, Hm = H.copy(), H.copy()
            Hp[i, j] += h
            Hm[i, j] -= h
            num_dH[i, j] = (L(Hp, W) - L(Hm, W)) / (2 * h)
    num_dW = np.zeros_like(W)
    for i in range(V):
        for j in range(d):
            Wp, Wm = W.copy(), W.copy()
            Wp[i, j] += h
            Wm[i, j] -= h
            num_dW[i, j] = (L(H, Wp) - L(H, Wm)) / (2 * h)
    for ana, num in ((dH, num_dH), (dW, num_dW)):
        rel = np.linalg.norm(ana - num) / max(np.linalg.norm(num), 1e-300)
        assert rel <= 1e-7, rel


# ------------------------------------------------ library routines (torch fp64)

def _torch_dense_loss(H, W, idx, logit, mask, tau):
    """Dense KL through torch library routines: kl_div(log_softmax(z/tau), P)."""
    Ht = torch.tensor(H, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    logq = torch.log_softmax((Ht @ Wt.T) / tau, dim=1)
    p = torch.softmax(torch.tensor(logit, dtype=torch.float64) / tau, dim=1)
    P = torch.zeros_like(logq).scatter_add_(1, torch.tensor(idx, dtype=torch.int64), p)
    kl = torch.nn.functional.kl_div(logq, P, reduction="none").sum(dim=1)
    m = torch.tensor(mask != 0, dtype=torch.float64)
    loss = (kl * m).sum() / m.sum()
    return loss, kl, Ht, Wt


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_against_torch_autograd(seed):
    rng = np.random.default_rng(seed)
    T, d, V, K = 9, 12, 40, 6
    tau = [1.0, 2.0, 0.7][seed]
    H, W, idx, logit, mask = _rand_problem(rng, T, d, V, K)
    loss_t, kl_t, Ht, Wt = _torch_dense_loss(H, W, idx, logit, mask, tau)
    (2.5 * loss_t).backward()
    loss, lse, kl = ok.forward(H, W, idx, logit, mask, tau)
    assert abs(loss - loss_t.item()) <= 1e-12 * max(1.0, abs(loss))
    np.testing.assert_allclose(kl, kl_t.detach().numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.tensor(H @ W.T / tau), dim=1).numpy(),
                               rtol=1e-13, atol=1e-13)
    dH, dW = ok.backward(H, W, idx, logit, mask, tau, 2.5)
    np.testing.assert_allclose(dH, Ht.grad.numpy(), rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-10, atol=1e-14)


def test_k1_is_cross_entropy():
    rng = np.random.default_rng(7)
    T, d, V = 11, 8, 50
    H, W, idx, logit, mask = _rand_problem(rng, T, d, V, 1, mask_p=1.0)
    for tau in (1.0, 3.0):
        _, _, kl = ok.forward(H, W, idx, logit, mask, tau)
        ce = torch.nn.functional.cross_entropy(torch.tensor(H @ W.T / tau), torch.tensor(idx[:, 0]),
                                               reduction="none").numpy()
        np.testing.assert_allclose(kl, ce, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ invariants

def test_kl_nonnegative():
    rng = np.random.default_rng(3)
    for K in (1, 5, 30):
        H, W, idx, logit, mask = _rand_problem(rng, 20, 16, 64, K)
        _, _, kl = ok.forward(H, W, idx, logit, mask, 1.3)
        assert (kl >= -1e-12).all()


@pytest.mark.parametrize("tau", [1.0, 2.0])
def test_teacher_equals_student_gives_zero(tau):
    rng = np.random.default_rng(4)
    T, d, V = 6, 5, 13
    H = rng.standard_normal((T, d))
    W = rng.standard_normal((V, d))
    z = H @ W.T
    idx = np.stack([rng.permutation(V) for _ in range(T)])
    logit = np.take_along_axis(z, idx, axis=1)
    mask = np.ones(T, np.uint8)
    loss, _, kl = ok.forward(H, W, idx, logit, mask, tau)
    assert np.abs(kl).max() < 1e-12 and abs(loss) < 1e-12
    G = ok.grad_logits(H, W, idx, logit, mask, tau)
    assert np.abs(G).max() < 1e-14


def test_shift_invariance():
    rng = np.random.default_rng(5)
    T, d, V, K, tau = 7, 6, 30, 5, 1.5
    H, W, idx, logit, mask = _rand_problem(rng, T, d, V, K)
    loss0, lse0, kl0 = ok.forward(H, W, idx, logit, mask, tau)
    dH0, dW0 = ok.backward(H, W, idx, logit, mask, tau)
    # a constant per teacher row
    c = rng.standard_normal((T, 1)) * 5
    loss1, _, kl1 = ok.forward(H, W, idx, logit + c, mask, tau)
    assert abs(loss1 - loss0) < 1e-12
    np.testing.assert_allclose(kl1, kl0, atol=1e-12)
    # a constant per student row: an extra feature column c_t in H and 1 in W
    c2 = rng.standard_normal(T) * 5
    H2 = np.concatenate([H, c2[:, None]], axis=1)
    W2 = np.concatenate([W, np.ones((V, 1))], axis=1)
    loss2, lse2, kl2 = ok.forward(H2, W2, idx, logit, mask, tau)
    assert abs(loss2 - loss0) < 1e-12
    np.testing.assert_allclose(lse2, lse0 + c2 / tau, atol=1e-12)
    dH2, dW2 = ok.backward(H2, W2, idx, logit, mask, tau)
    np.testing.assert_allclose(dH2[:, :d], dH0, atol=1e-14)
    np.testing.assert_allclose(dW2[:, :d], dW0, atol=1e-14)


def test_gradient_rows_sum_to_zero():
    rng = np.random.default_rng(6)
    H, W, idx, logit, mask = _rand_problem(rng, 10, 9, 33, 4)
    G = ok.grad_logits(H, W, idx, logit, mask, 1.0, 2.0)
    assert np.abs(G.sum(axis=1)).max() < 1e-15
    _, dW = ok.backward(H, W, idx, logit, mask, 1.0, 2.0)
    assert np.abs(dW.sum(axis=0)).max() < 1e-14


def test_dense_grid_equals_gathered():
    rng = np.random.default_rng(8)
    H, W, idx, logit, mask = _rand_problem(rng, 12, 7, 45, 9)
    logq, _ = ok.student_log_softmax(H, W, 1.2)
    p = ok.teacher_probs(logit, 1.2)
    np.testing.assert_allclose(ok.dense_kl(logq, ok.dense_teacher(idx, p, 45)),
                               ok.token_kl(logq, idx, p), rtol=1e-12, atol=1e-13)


def test_permutation_over_k():
    rng = np.random.default_rng(9)
    H, W, idx, logit, mask = _rand_problem(rng, 8, 6, 25, 5)
    perm = rng.permutation(5)
    a = ok.forward(H, W, idx, logit, mask, 1.0)
    b = ok.forward(H, W, idx[:, perm], logit[:, perm], mask, 1.0)
    assert abs(a[0] - b[0]) < 1e-13
    np.testing.assert_allclose(ok.backward(H, W, idx, logit, mask, 1.0)[1],
                               ok.backward(H, W, idx[:, perm], logit[:, perm], mask, 1.0)[1], atol=1e-15)


def test_mask_invariance():
    rng = np.random.default_rng(10)
    H, W, idx, logit, mask = _rand_problem(rng, 10, 6, 20, 4, mask_p=0.5)
    H2 = H.copy()
    H2[mask == 0] = rng.standard_normal(((mask == 0).sum(), 6)) * 10
    a, b = ok.forward(H, W, idx, logit, mask, 1.0), ok.forward(H2, W, idx, logit, mask, 1.0)
    assert abs(a[0] - b[0]) < 1e-13
    dHa, dWa = ok.backward(H, W, idx, logit, mask, 1.0)
    dHb, dWb = ok.backward(H2, W, idx, logit, mask, 1.0)
    np.testing.assert_allclose(dWa, dWb, atol=1e-15)
    np.testing.assert_allclose(dHa[mask != 0], dHb[mask != 0], atol=1e-15)
    assert not dHb[mask == 0].any()


def test_all_masked():
    rng = np.random.default_rng(11)
    H, W, idx, logit, _ = _rand_problem(rng, 4, 5, 9, 2)
    mask = np.zeros(4, np.uint8)
    assert ok.forward(H, W, idx, logit, mask, 1.0)[0] == 0.0
    dH, dW = ok.backward(H, W, idx, logit, mask, 1.0)
    assert not dH.any() and not dW.any()


def test_neg_inf_teacher_logit_contributes_nothing():
    rng = np.random.default_rng(12)
    H, W, idx, logit, mask = _rand_problem(rng, 5, 4, 15, 3, mask_p=1.0)
    logit2 = np.concatenate([logit, np.full((5, 1), -np.inf)], axis=1)
    extra = np.array([[v for v in range(15) if v not in row][0] for row in idx])
    idx2 = np.concatenate([idx, extra[:, None]], axis=1)
    a, b = ok.forward(H, W, idx, logit, mask, 1.0), ok.forward(H, W, idx2, logit2, mask, 1.0)
    assert abs(a[0] - b[0]) < 1e-13
    np.testing.assert_allclose(ok.backward(H, W, idx, logit, mask, 1.0)[0],
                               ok.backward(H, W, idx2, logit2, mask, 1.0)[0], atol=1e-15)


def test_out_of_range_index_rejected():
    rng = np.random.default_rng(13)
    H, W, idx, logit, mask = _rand_problem(rng, 3, 4, 10, 2)
    idx[1, 0] = 10
    with pytest.raises(ValueError):
        ok.forward(H, W, idx, logit, mask, 1.0)


# ------------------------------------------------ sampled (large-size) helpers

def test_sampled_helpers_match_dense():
    rng = np.random.default_rng(14)
    T, d, V, K, tau = 40, 10, 70, 6, 1.4
    H, W, idx, logit, mask = _rand_problem(rng, T, d, V, K)
    loss, lse, kl = ok.forward(H, W, idx, logit, mask, tau)
    dH, dW = ok.backward(H, W, idx, logit, mask, tau, 0.9)
    np.testing.assert_allclose(ok.lse_rows(H, W, tau, rows_per_block=7), lse, rtol=1e-14)
    rows = np.array([0, 5, 39])
    G = ok.grad_logits(H[rows], W, idx[rows], logit[rows], mask[rows], tau, 0.9,
                       n_total=ok.mask_count(mask))
    np.testing.assert_allclose(G @ W, dH[rows], rtol=1e-12, atol=1e-16)
    vs = np.array([0, idx[3, 2], 69])
    np.testing.assert_allclose(ok.dW_rows(H, W, idx, logit, mask, tau, vs, lse, 0.9), dW[vs],
                               rtol=1e-12, atol=1e-16)


# ---------------------------------------------------------------- bf16 widening

def test_bf16_widening_exact():
    bits = np.array([0x3F80, 0xC000, 0x7F80, 0xFF80, 0x0001, 0x8000, 0x3E80], dtype=np.uint16)
    want = [1.0, -2.0, np.inf, -np.inf, 2.0 ** -133, -0.0, 0.25]
    got = ok.bf16_bits_to_f64(bits)
    for g_, w_ in zip(got, want):
        assert g_ == w_ and math.copysign(1, g_) == math.copysign(1, w_)
    rnd = np.random.default_rng(0).integers(0, 2 ** 16, 4096).astype(np.uint16)
    rnd = rnd[(rnd & 0x7F80) != 0x7F80]  # drop inf/nan patterns
    lib = torch.from_numpy(rnd.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ok.bf16_bits_to_f64(rnd), lib)


# ------------------------------------------------------------ planted mistakes

def _pins_pass(mod) -> bool:
    """Run a subset of the pins above against a (possibly mutated) oracle."""
    try:
        for case in _golden_cases():
            tau, g = _ev(case["tau"]), _ev(case["grad_loss"])
            H, W = _evm(case["H"]), _evm(case["W"])
            idx = np.array(case["topk_idx"])
            logit = _evm(case["topk_logit"])
            mask = np.array(case["mask"], dtype=np.uint8)
            loss = mod.forward(H, W, idx, logit, mask, tau)[0]
            if abs(loss - _ev(case["expect"]["loss"])) > 1e-12:
                return False
            dH, dW = mod.backward(H, W, idx, logit, mask, tau, g)
            if np.abs(dH - _evm(case["expect"]["dH"])).max() > 1e-12:
                return False
            if np.abs(dW - _evm(case["expect"]["dW"])).max() > 1e-12:
                return False
        rng = np.random.default_rng(1)
        H, W, idx, logit, mask = _rand_problem(rng, 9, 12, 40, 6)
        loss_t, _, Ht, Wt = _torch_dense_loss(H, W, idx, logit, mask, 2.0)
        loss_t.backward()
        if abs(mod.forward(H, W, idx, logit, mask, 2.0)[0] - loss_t.item()) > 1e-10:
            return False
        dH, dW = mod.backward(H, W, idx, logit, mask, 2.0)
        return np.allclose(dH, Ht.grad.numpy(), rtol=1e-9) and np.allclose(dW, Wt.grad.numpy(), rtol=1e-9)
    except Exception:  # noqa: BLE001 - a planted mistake that raises fails the pins too
        return False


MUTANTS = {
    "teacher_without_tau": ("teacher_probs",
                            lambda orig: (lambda l, tau: orig(l, 1.0))),
    "student_without_tau": ("student_log_softmax",
                            lambda orig: (lambda H, W, tau: orig(H, W, 1.0))),
    "dropped_entropy_term": ("_xlogx_terms", lambda orig: (lambda p: np.zeros_like(p))),
    "gradient_sign_flipped": ("grad_logits",
                              lambda orig: (lambda *a, **k: -orig(*a, **k))),
    "gradient_missing_tau": ("grad_logits",
                             lambda orig: (lambda H, W, i, l, m, tau, g=1.0, n_total=None:
                                           orig(H, W, i, l, m, tau, g, n_total) * tau)),
    "teacher_not_renormalised": ("teacher_probs",
                                 lambda orig: (lambda l, tau: np.exp(np.asarray(l) / tau))),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    assert _pins_pass(ok), "pins must pass on the real oracle"
    attr, make = MUTANTS[name]
    monkeypatch.setattr(ok, attr, make(getattr(ok, attr)))
    assert not _pins_pass(ok), "planted mistake %s went undetected" % name


def test_planted_transposed_backward_is_caught(monkeypatch):
    real = ok.backward

    def transposed(H, W, i, l, m, tau, g=1.0):
        G = ok.grad_logits(H, W, i, l, m, tau, g)
        return G @ np.asarray(W), (np.asarray(H).T @ G).T[:, ::-1]

    monkeypatch.setattr(ok, "backward", transposed)
    assert not _pins_pass(ok)
    monkeypatch.setattr(ok, "backward", real)
    assert _pins_pass(ok)


def test_forward_all_rows_matches_forward():
    rng = np.random.default_rng(15)
    H, W, idx, logit, mask = _rand_problem(rng, 50, 8, 60, 5, mask_p=1.0)
    _, lse, kl = ok.forward(H, W, idx, logit, mask, 1.3)
    lse2, kl2 = ok.forward_all_rows(H, W, idx, logit, 1.3, rows_per_block=7, workers=3)
    np.testing.assert_allclose(lse2, lse, rtol=1e-14)
    np.testing.assert_allclose(kl2, kl, rtol=1e-12, atol=1e-14)
