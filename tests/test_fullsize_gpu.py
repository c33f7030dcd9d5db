"""Full-size parity: the workloads' real shapes, in the launch configuration
the benchmark uses, against the fp64 oracle.

Two kinds of check per workload:

* full mask (the benchmark's data): lse and per-token KL on sampled token rows
  (tile and sequence boundaries plus random rows), dH on sampled rows, masked
  dH rows exactly zero, and loss == mean of the per-token KL over the mask.
* sparse mask (only a sampled token set S counts, m_t = 0 elsewhere): the
  kernels run the identical full-size grid, and the oracle, which then needs
  only the rows of S, gives the exact loss and EVERY row of dW.
"""
import numpy as np
import pytest
import torch

import oracle.kl_oracle as ok
from lm_head_top_gb300.inputs import WORKLOADS, make_inputs
from tests._helpers import GRAD_REL_L2, LOSS_RTOL, LSE_ATOL, max_err_counted, rel_l2

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def kdkl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_top_gb300 import kdkl as m
    m.load()
    return m


def _rows(T, n, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 129, 255, 256, T // 2, T - 129, T - 128, T - 2, T - 1]
    fixed = [r for r in fixed if 0 <= r < T]
    rest = rng.choice(T, size=max(n - len(fixed), 0), replace=False)
    return np.unique(np.concatenate([fixed, rest]).astype(np.int64))


class Run:
    """One forward + backward on the GPU; results stay on the device."""

    def __init__(self, kdkl, g, w, mask, chunk=None):
        self.loss, self.lse, self.kl = kdkl.kd_kl_forward(
            g["H"], g["W"], g["topk_idx"], g["topk_logit"], mask, temperature=w.tau,
            chunk=chunk or w.chunk, want_token_kl=True)
        self.dH, self.dW = kdkl.kd_kl_backward(
            g["H"], g["W"], g["topk_idx"], g["topk_logit"], mask, self.lse, temperature=w.tau,
            chunk=chunk or w.chunk, grad_loss=1.0)
        torch.cuda.synchronize()

    def rows(self, name, rows):
        t = getattr(self, name)
        return t[torch.as_tensor(rows, device=t.device)].float().cpu().numpy().astype(np.float64)


class _Rows:
    """H widened to fp64 on demand, one row set at a time (H can be GBs)."""

    def __init__(self, H_bf16):
        self.bits = H_bf16.view(torch.int16).numpy()

    def __getitem__(self, rows):
        return ok.bf16_bits_to_f64(self.bits[np.asarray(rows)])


def _oracle_np(x):
    W = ok.bf16_bits_to_f64(x["W"].view(torch.int16).numpy())
    return (_Rows(x["H"]), W, x["topk_idx"].numpy().astype(np.int64),
            x["topk_logit"].numpy().astype(np.float64))


def check_full_mask(kdkl, w, x, g, Hn, Wn, idx, lg, chunk=None, n_rows=64, seed=0):
    mask = x["mask"].numpy()
    run = Run(kdkl, g, w, g["mask"], chunk)
    rows = _rows(w.T, n_rows, seed)
    r_loss, r_lse, r_kl = ok.forward(Hn[rows], Wn, idx[rows], lg[rows], mask[rows], w.tau)
    assert max_err_counted(run.rows("lse", rows), r_lse, mask[rows]) <= LSE_ATOL
    assert max_err_counted(run.rows("kl", rows), r_kl, mask[rows]) <= 1e-3 * max(1.0, np.abs(r_kl).max())
    n = int(mask.sum())
    G = ok.grad_logits(Hn[rows], Wn, idx[rows], lg[rows], mask[rows], w.tau, 1.0, n_total=n)
    dH = run.rows("dH", rows)
    assert rel_l2(dH, G @ Wn) <= GRAD_REL_L2
    assert not dH[mask[rows] == 0].any()
    # loss is the mean of the (device) per-token KL over the mask
    kl_all = run.kl.double().cpu().numpy()
    assert abs(run.loss.item() - kl_all[mask != 0].mean()) <= 1e-5 * abs(run.loss.item())
    # Every row of G sums to zero over the vocabulary (q and P are both
    # distributions), so the columns of dW = G^T H sum to zero: a check on
    # every row of the full-size dW. What remains is the bf16 rounding of G
    # (~1e-3 of |dW|); a dropped tile or slab leaves several per cent.
    # Summed in fp64 over 256-row blocks: a few MB of temporaries.
    colsum = torch.zeros(run.dW.shape[1], dtype=torch.float64, device=run.dW.device)
    sq = torch.zeros((), dtype=torch.float64, device=run.dW.device)
    for r0 in range(0, run.dW.shape[0], 256):
        blk = run.dW[r0:r0 + 256].double()
        colsum += blk.sum(0)
        sq += (blk * blk).sum()
        del blk
    assert (torch.linalg.vector_norm(colsum) / sq.sqrt()).item() <= 1e-2
    return run


def check_sparse_mask(kdkl, w, x, g, Hn, Wn, idx, lg, chunk=None, n_tokens=192, seed=1):
    T = w.T
    S = _rows(T, n_tokens, seed)
    base = x["mask"].numpy()
    sparse = np.zeros(T, dtype=np.uint8)
    sparse[S] = base[S]
    if sparse.sum() == 0:
        sparse[S[0]] = 1
    run = Run(kdkl, g, w, torch.from_numpy(sparse).to(g["H"].device), chunk)
    r_loss, r_lse, r_kl = ok.forward(Hn[S], Wn, idx[S], lg[S], sparse[S], w.tau)
    assert abs(run.loss.item() - r_loss) <= LOSS_RTOL * abs(r_loss)
    assert max_err_counted(run.rows("lse", S), r_lse, sparse[S]) <= LSE_ATOL
    G = ok.grad_logits(Hn[S], Wn, idx[S], lg[S], sparse[S], w.tau, 1.0, n_total=int(sparse.sum()))
    assert rel_l2(run.rows("dH", S), G @ Wn) <= GRAD_REL_L2
    dW = run.dW.double().cpu().numpy()
    assert rel_l2(dW, G.T @ Hn[S]) <= GRAD_REL_L2
    # rows outside S got nothing
    other = np.setdiff1d(_rows(T, 64, seed + 7), S)
    assert not run.rows("dH", other).any()
    return run


def _inputs(name, **over):
    w = WORKLOADS[name].with_(**over) if over else WORKLOADS[name]
    x = make_inputs(w, seed=0, topk_device="cuda")
    g = {k: v.cuda() for k, v in x.items()}
    return w, x, g


def test_gptoss20b_32k(kdkl):
    """The benchmark's workload, seed and launch configuration."""
    w, x, g = _inputs("gptoss20b_32k")
    Hn, Wn, idx, lg = _oracle_np(x)
    check_full_mask(kdkl, w, x, g, Hn, Wn, idx, lg)
    check_sparse_mask(kdkl, w, x, g, Hn, Wn, idx, lg)


def test_llama3b_8k(kdkl):
    w, x, g = _inputs("llama3b_8k")
    Hn, Wn, idx, lg = _oracle_np(x)
    check_full_mask(kdkl, w, x, g, Hn, Wn, idx, lg)
    check_sparse_mask(kdkl, w, x, g, Hn, Wn, idx, lg)


@pytest.mark.parametrize("K", [1, 20, 100, 512])
def test_padded_4x8k_sweep(kdkl, K):
    """Batch 4 x 8192 with the last 20 % of each sequence masked; tau and chunk
    swept. The forward is chunk-independent (bitwise) and the gradients agree
    across chunk sizes."""
    w0, x, g = _inputs("padded_4x8k", K=K)
    Hn, Wn, idx, lg = _oracle_np(x)
    for tau in (1.0, 2.0):
        w = w0.with_(tau=tau)
        runs = [check_full_mask(kdkl, w, x, g, Hn, Wn, idx, lg, chunk=c, n_rows=40, seed=K)
                for c in (512, 1024, 4096)]
        for r in runs[1:]:
            assert r.loss.item() == runs[0].loss.item()
            assert rel_l2(r.dW.double().cpu().numpy(), runs[0].dW.double().cpu().numpy()) < 1e-4
            assert rel_l2(r.dH.double().cpu().numpy(), runs[0].dH.double().cpu().numpy()) < 1e-2
        del runs
        if K == 100:
            check_sparse_mask(kdkl, w, x, g, Hn, Wn, idx, lg, chunk=1024, seed=int(tau))


def test_toyproj_256k_memory_linear(kdkl):
    """256K tokens: token-chunked backward (T > V); peak memory has no T x V term."""
    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats()
    w, x, g = _inputs("toyproj_256k")
    base = torch.cuda.memory_allocated()
    Hn, Wn, idx, lg = _oracle_np(x)
    run = check_full_mask(kdkl, w, x, g, Hn, Wn, idx, lg, n_rows=48)
    peak = torch.cuda.max_memory_allocated()
    T, d, V, K = w.T, w.d, w.V, w.K
    ws = max(kdkl.kd_kl_workspace_size(T, d, V, K, 1.0, w.chunk, 0),
             kdkl.kd_kl_workspace_size(T, d, V, K, 1.0, w.chunk, 1))
    outputs = T * 4 * 2 + T * d * 2 + V * d * 4  # lse, token_kl, dH, dW
    assert peak <= base + outputs + ws + (64 << 20), (peak, base, outputs, ws)
    assert peak < 0.25 * T * V * 4  # far below one fp32 logit grid
    del run
    check_sparse_mask(kdkl, w, x, g, Hn, Wn, idx, lg, n_tokens=128)
