"""fp64 CPU oracle for the fused chunked KL distillation loss.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers. The product path (the CUDA
library and its Python binding) never imports, calls or links anything here,
and nothing here imports the product. Inputs reach both sides from the seeded
generator, which holds none of this arithmetic.

What it computes follows the pages' statement of the method ("Making
knowledge distillation cheap enough to run at scale", section "Two system
changes"; the same method in "Efficient knowledge distillation for LLMs:
offline top-K logits and a fused chunked KL loss", section "Two systemic
changes for scalable distillation"):

* the teacher is an offline cache of its top-K (id, logit) pairs per token
  (the "Offline distillation" paragraph of that section);
* the loss is the KL divergence between the teacher distribution and the
  student's full-vocabulary distribution, whose logits are the student's
  output projection z = H W^T (the "Fused, chunked KL loss" paragraph; the
  dense KL is the textbook form those bullets use as the correctness
  baseline, and the three offline variants are stated to be mathematically
  equivalent);
* the closed-form gradient is named but never printed on the pages; it is
  derived here from the definition.

Readings taken where the pages are silent (each is pinned by a test):

1. Teacher: p_{t,k} = softmax_k(topk_logit_{t,k} / tau), renormalised over the
   K cached entries (a -inf logit gives p = 0).
2. Student: log q_{t,v} = z_{t,v}/tau - lse_t with lse_t = log sum_v exp(z_{t,v}/tau),
   over the FULL vocabulary (not renormalised over the K ids).
3. Direction: forward KL(p || q), per entry:
   KL_t = sum_k p_{t,k} (log p_{t,k} - log q_{t, idx_{t,k}}), with 0 log 0 = 0.
4. No tau^2 factor.
5. loss = sum_t m_t KL_t / N with N = sum_t m_t (mask m_t in {0,1}); loss = 0
   when N = 0.
6. dL/dz_{t,v} = m_t (q_{t,v} - P_{t,v}) / (tau N), where P scatter-adds the
   K teacher probabilities of row t into a dense vocabulary row (duplicate ids
   add up). The upstream gradient g = dL_outer/dloss scales it.
7. dH = G W and dW = G^T H with G = g dL/dz.

The only "blocking" is over rows (tokens), which the definition treats
independently; no step is fused or reordered.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16/int16 array) to float64:
    a bf16 value is the upper half of the float32 with the same bits."""
    b = np.asarray(bits).view(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def teacher_probs(topk_logit, tau: float) -> np.ndarray:
    """Reading 1: p_{t,k} = exp(l_{t,k}/tau) / sum_j exp(l_{t,j}/tau)."""
    a = np.asarray(topk_logit, dtype=np.float64) / tau
    amax = np.max(a, axis=1, keepdims=True)
    e = np.exp(a - amax)
    return e / np.sum(e, axis=1, keepdims=True)


def student_logits(H, W) -> np.ndarray:
    """The student's output projection z = H W^T (dense tokens x vocab grid)."""
    return np.asarray(H, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def student_log_softmax(H, W, tau: float):
    """Reading 2: returns (log q [T,V], lse [T]) with lse_t = log sum_v e^{z_{t,v}/tau}."""
    zt = student_logits(H, W) / tau
    zmax = np.max(zt, axis=1, keepdims=True)
    lse = zmax[:, 0] + np.log(np.sum(np.exp(zt - zmax), axis=1))
    return zt - lse[:, None], lse


def _xlogx_terms(p: np.ndarray) -> np.ndarray:
    """p log p with the convention 0 log 0 = 0."""
    safe = np.where(p > 0, p, 1.0)
    return np.where(p > 0, p * np.log(safe), 0.0)


def token_kl(logq, topk_idx, p) -> np.ndarray:
    """Reading 3: KL_t = sum_k p_{t,k} (log p_{t,k} - log q_{t, idx_{t,k}})."""
    logq_at = np.take_along_axis(logq, np.asarray(topk_idx, dtype=np.int64), axis=1)
    cross = np.where(p > 0, p * logq_at, 0.0)
    return np.sum(_xlogx_terms(p), axis=1) - np.sum(cross, axis=1)


def mask_count(mask) -> int:
    return int(np.count_nonzero(np.asarray(mask)))


def check_indices(topk_idx, V: int) -> None:
    idx = np.asarray(topk_idx)
    if idx.size and (idx.min() < 0 or idx.max() >= V):
        raise ValueError("topk_idx outside [0, V)")


def forward(H, W, topk_idx, topk_logit, mask, tau: float):
    """Returns (loss, lse [T], token_kl [T]) from the dense definition."""
    check_indices(topk_idx, np.asarray(W).shape[0])
    logq, lse = student_log_softmax(H, W, tau)
    p = teacher_probs(topk_logit, tau)
    kl = token_kl(logq, topk_idx, p)
    m = np.asarray(mask) != 0
    n = int(np.count_nonzero(m))
    loss = float(np.sum(kl[m]) / n) if n else 0.0
    return loss, lse, kl


def dense_teacher(topk_idx, p, V: int) -> np.ndarray:
    """Reading 6's P: the K teacher probabilities of each row scattered into a
    dense vocabulary row (the 'dense KL' grid), duplicate ids adding up."""
    T = p.shape[0]
    P = np.zeros((T, V), dtype=np.float64)
    rows = np.repeat(np.arange(T), p.shape[1])
    np.add.at(P, (rows, np.asarray(topk_idx, dtype=np.int64).ravel()), p.ravel())
    return P


def dense_kl(logq, P) -> np.ndarray:
    """The pages' dense KL: sum over the whole vocabulary of P (log P - log q)."""
    return np.sum(_xlogx_terms(P), axis=1) - np.sum(np.where(P > 0, P * logq, 0.0), axis=1)


def grad_logits(H, W, topk_idx, topk_logit, mask, tau: float, grad_loss: float = 1.0,
                n_total: int | None = None) -> np.ndarray:
    """Reading 6/7: G_{t,v} = g m_t (q_{t,v} - P_{t,v}) / (tau N) for the given rows.

    ``n_total`` is N over the whole batch when the rows passed are a subset."""
    V = np.asarray(W).shape[0]
    logq, _ = student_log_softmax(H, W, tau)
    q = np.exp(logq)
    P = dense_teacher(topk_idx, teacher_probs(topk_logit, tau), V)
    m = (np.asarray(mask) != 0).astype(np.float64)
    n = mask_count(mask) if n_total is None else int(n_total)
    if n == 0:
        return np.zeros_like(q)
    return (q - P) * (grad_loss * m / (tau * n))[:, None]


def backward(H, W, topk_idx, topk_logit, mask, tau: float, grad_loss: float = 1.0):
    """Returns (dH [T,d], dW [V,d]) in fp64: dH = G W, dW = G^T H."""
    check_indices(topk_idx, np.asarray(W).shape[0])
    G = grad_logits(H, W, topk_idx, topk_logit, mask, tau, grad_loss)
    return G @ np.asarray(W, dtype=np.float64), G.T @ np.asarray(H, dtype=np.float64)


def lse_rows(H, W, tau: float, rows_per_block: int = 256) -> np.ndarray:
    """lse_t for every row of H, one block of rows at a time (rows are
    independent in the definition)."""
    H = np.asarray(H)
    out = np.empty(H.shape[0], dtype=np.float64)
    for r0 in range(0, H.shape[0], rows_per_block):
        out[r0:r0 + rows_per_block] = student_log_softmax(H[r0:r0 + rows_per_block], W, tau)[1]
    return out


def forward_all_rows(H, W, topk_idx, topk_logit, tau: float, rows_per_block: int = 128,
                     workers: int | None = None):
    """(lse [T], token_kl [T]) for every row: ``forward`` applied to blocks of
    rows, the blocks run by a thread pool (numpy releases the GIL in BLAS and
    in the elementwise steps). Each row's arithmetic is exactly ``forward``'s."""
    import concurrent.futures as cf
    import os

    H = np.asarray(H)
    W = np.asarray(W, dtype=np.float64)
    T = H.shape[0]
    lse = np.empty(T, dtype=np.float64)
    kl = np.empty(T, dtype=np.float64)
    ones = np.ones(T, dtype=np.uint8)

    def block(r0):
        r1 = min(r0 + rows_per_block, T)
        _, l, k = forward(H[r0:r1], W, topk_idx[r0:r1], topk_logit[r0:r1], ones[r0:r1], tau)
        lse[r0:r1] = l
        kl[r0:r1] = k

    n = workers or max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(n) as ex:
        list(ex.map(block, range(0, T, rows_per_block)))
    return lse, kl


def dW_rows(H, W, topk_idx, topk_logit, mask, tau: float, vocab_rows, lse,
            grad_loss: float = 1.0) -> np.ndarray:
    """dW[v, :] = sum_t G_{t,v} H_t for the listed vocabulary rows v, given the
    full lse [T] (from ``lse_rows``). Same definition as ``backward``,
    evaluated only on the requested columns of G."""
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    vs = np.asarray(vocab_rows, dtype=np.int64)
    zt = (H @ W[vs].T) / tau  # [T, |vs|]
    q = np.exp(zt - np.asarray(lse)[:, None])
    p = teacher_probs(topk_logit, tau)
    idx = np.asarray(topk_idx, dtype=np.int64)
    P = np.zeros_like(q)
    for j, v in enumerate(vs):
        P[:, j] = np.sum(np.where(idx == v, p, 0.0), axis=1)
    m = (np.asarray(mask) != 0).astype(np.float64)
    n = mask_count(mask)
    if n == 0:
        return np.zeros((len(vs), H.shape[1]))
    G = (q - P) * (grad_loss * m / (tau * n))[:, None]
    return G.T @ H


# --------------------------------------------------------------------------
# Offline teacher cache: the top-K (id, logit) pairs of each row of z = H W^T.
# ("Making knowledge distillation cheap enough to run at scale", section "Two
# system changes": compute the teacher's output once and cache the 100 most
# likely tokens per position.) Order: logit descending, ties by smaller id.

def topk_logits(H, W, K: int):
    """(ids [T,K] int64, logits [T,K] fp64) from the dense fp64 grid z = H W^T,
    each row sorted by (logit descending, id ascending)."""
    z = student_logits(H, W)
    T, V = z.shape
    if not 1 <= K <= V:
        raise ValueError("need 1 <= K <= V")
    ids = np.empty((T, K), dtype=np.int64)
    for t in range(T):
        # lexsort: last key is primary; -z descending, then id ascending
        order = np.lexsort((np.arange(V), -z[t]))
        ids[t] = order[:K]
    return ids, np.take_along_axis(z, ids, axis=1)


# --------------------------------------------------------------------------
# Loss variant: the soft KL term mixed with a hard-label cross-entropy.
# The pages report ablations over the choice of loss without printing one;
# this is the standard distillation mix, read plainly:
#   loss_t = alpha * c * KL_t(tau) + (1 - alpha) * CE_t,
#   CE_t   = logsumexp_v z_{t,v} - z_{t, y_t}          (temperature 1),
#   c      = tau^2 when scale_tau_sq else 1.
# dL/dz = m_t / N * [alpha c (q_tau - P) / tau + (1 - alpha) (q_1 - onehot(y_t))].

def forward_mixed(H, W, topk_idx, topk_logit, mask, tau: float, alpha: float,
                  scale_tau_sq: bool, labels):
    """Returns (loss, lse_tau [T], lse_1 [T], token_loss [T])."""
    check_indices(topk_idx, np.asarray(W).shape[0])
    check_indices(np.asarray(labels)[:, None], np.asarray(W).shape[0])
    logq, lse = student_log_softmax(H, W, tau)
    kl = token_kl(logq, topk_idx, teacher_probs(topk_logit, tau))
    logq1, lse1 = student_log_softmax(H, W, 1.0)
    ce = -np.take_along_axis(logq1, np.asarray(labels, dtype=np.int64)[:, None], axis=1)[:, 0]
    c = tau * tau if scale_tau_sq else 1.0
    tok = alpha * c * kl + (1.0 - alpha) * ce
    m = np.asarray(mask) != 0
    n = int(np.count_nonzero(m))
    loss = float(np.sum(tok[m]) / n) if n else 0.0
    return loss, lse, lse1, tok


def backward_mixed(H, W, topk_idx, topk_logit, mask, tau: float, alpha: float,
                   scale_tau_sq: bool, labels, grad_loss: float = 1.0):
    """Returns (dH, dW) of grad_loss * forward_mixed's loss."""
    V = np.asarray(W).shape[0]
    logq, _ = student_log_softmax(H, W, tau)
    P = dense_teacher(topk_idx, teacher_probs(topk_logit, tau), V)
    logq1, _ = student_log_softmax(H, W, 1.0)
    Y = np.zeros_like(logq1)
    Y[np.arange(Y.shape[0]), np.asarray(labels, dtype=np.int64)] = 1.0
    c = tau * tau if scale_tau_sq else 1.0
    m = (np.asarray(mask) != 0).astype(np.float64)
    n = mask_count(mask)
    if n == 0:
        return np.zeros_like(np.asarray(H, dtype=np.float64)), np.zeros_like(np.asarray(W, dtype=np.float64))
    G = (alpha * c * (np.exp(logq) - P) / tau + (1.0 - alpha) * (np.exp(logq1) - Y))
    G = G * (grad_loss * m / n)[:, None]
    return G @ np.asarray(W, dtype=np.float64), G.T @ np.asarray(H, dtype=np.float64)


# --------------------------------------------------------------------------
# Reverse KL restricted to the cached ids (a loss-choice variant): both the
# student and the teacher are renormalised over the row's K cached entries;
# entries whose teacher logit is -inf are outside the support and dropped.
#   qt_k = softmax_k(z[t, idx_k] / tau),  p_k = softmax_k(topk_logit_k / tau)
#   RKL_t = sum_k qt_k (log qt_k - log p_k),   loss = sum_t m_t RKL_t / N
# d RKL_t / d z[t, idx_k] = qt_k (log qt_k - log p_k - RKL_t) / tau

def _support_logsoftmax(a, keep):
    a = np.where(keep, a, -np.inf)
    amax = np.max(a, axis=1, keepdims=True)
    lse = amax[:, 0] + np.log(np.sum(np.where(keep, np.exp(a - amax), 0.0), axis=1))
    return np.where(keep, a - lse[:, None], -np.inf)


def reverse_kl_forward(H, W, topk_idx, topk_logit, mask, tau: float):
    """Returns (loss, token_rkl [T], z_at [T,K]) with z_at = z[t, idx_k]."""
    check_indices(topk_idx, np.asarray(W).shape[0])
    idx = np.asarray(topk_idx, dtype=np.int64)
    z_at = np.take_along_axis(student_logits(H, W), idx, axis=1)
    logit = np.asarray(topk_logit, dtype=np.float64)
    keep = np.isfinite(logit)
    logqt = _support_logsoftmax(z_at / tau, keep)
    logp = _support_logsoftmax(logit / tau, keep)
    qt = np.where(keep, np.exp(logqt), 0.0)
    with np.errstate(invalid="ignore"):  # -inf - -inf only in dropped entries
        rkl = np.sum(np.where(keep, qt * (logqt - logp), 0.0), axis=1)
    m = np.asarray(mask) != 0
    n = int(np.count_nonzero(m))
    return (float(np.sum(rkl[m]) / n) if n else 0.0), rkl, z_at


def reverse_kl_grad_z(H, W, topk_idx, topk_logit, mask, tau: float):
    """[T,K] derivative of reverse_kl_forward's loss with respect to the
    student logit z[t, idx_k] (0 for entries outside the support)."""
    idx = np.asarray(topk_idx, dtype=np.int64)
    _, rkl, z_at = reverse_kl_forward(H, W, idx, topk_logit, mask, tau)
    logit = np.asarray(topk_logit, dtype=np.float64)
    keep = np.isfinite(logit)
    logqt = _support_logsoftmax(z_at / tau, keep)
    logp = _support_logsoftmax(logit / tau, keep)
    qt = np.where(keep, np.exp(logqt), 0.0)
    m = (np.asarray(mask) != 0).astype(np.float64)
    n = mask_count(mask)
    if n == 0:
        return np.zeros(idx.shape)
    with np.errstate(invalid="ignore"):  # -inf - -inf only in dropped entries
        gk = np.where(keep, qt * (logqt - logp - rkl[:, None]), 0.0) / tau
    return gk * (m / n)[:, None]


def reverse_kl_backward(H, W, topk_idx, topk_logit, mask, tau: float, grad_loss: float = 1.0):
    """Returns (dH, dW) of grad_loss * reverse_kl_forward's loss."""
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = np.asarray(topk_idx, dtype=np.int64)
    gk = grad_loss * reverse_kl_grad_z(H, W, idx, topk_logit, mask, tau)
    G = np.zeros((H.shape[0], W.shape[0]))
    np.add.at(G, (np.repeat(np.arange(H.shape[0]), idx.shape[1]), idx.ravel()), gk.ravel())
    return G @ W, G.T @ H
