"""The backward that reuses the forward's prepared teacher rows
(kd_kl_backward_reuse), and the teacher-prep kernel's two key widths.

The reuse path must give exactly the results of the backward that prepares
the teacher rows itself (same sorted rows, same N, same kernels after that),
and both must match the fp64 oracle. A forward workspace that was not filled
for the same problem is refused."""
import os

import numpy as np
import pytest
import torch

import oracle.kl_oracle as ok
from lm_head_top_gb300.inputs import WORKLOADS, make_inputs
from tests._helpers import GRAD_REL_L2, LOSS_RTOL, rel_l2, to_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kdkl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_top_gb300 import kdkl as m
    m.load()
    return m


def _run(kdkl, x, tau, chunk, reuse, bwd_chunk=None, grad_loss=1.0):
    g = {k: v.cuda() for k, v in x.items()}
    T, d = g["H"].shape
    V, K = g["W"].shape[0], g["topk_idx"].shape[1]
    ws_f = torch.empty(kdkl.kd_kl_workspace_size(T, d, V, K, tau, chunk, 0), dtype=torch.uint8,
                       device="cuda")
    loss, lse, _ = kdkl.kd_kl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"],
                                      temperature=tau, chunk=chunk, workspace=ws_f)
    dH, dW = kdkl.kd_kl_backward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], lse,
                                 temperature=tau, chunk=bwd_chunk or chunk, grad_loss=grad_loss,
                                 fwd_workspace=ws_f if reuse else None)
    torch.cuda.synchronize()
    assert kdkl.kd_kl_check_status(ws_f) == 0
    return loss.item(), dH.cpu(), dW.cpu()


@pytest.mark.parametrize("shape", [
    # T, d, V, K, chunk, tau, pad
    (256, 256, 4096, 16, 64, 1.0, 0.0),
    (131, 72, 1000, 7, 50, 2.0, 0.25),      # ragged, vocabulary slabs
    (700, 64, 300, 5, 200, 1.0, 0.2),       # token chunks (T > V)
    (40, 48, 600, 512, 7, 1.0, 0.0),        # K = 512: 32 lanes x 16 entries per row
    (90, 32, 700, 200, 30, 0.7, 0.1),       # K = 200: 32 lanes x 8
    (33, 16, 64, 1, 8, 1.0, 0.0),           # K = 1
    (64, 32, 48, 48, 16, 0.5, 0.0),         # K = V, K % 4 == 0
])
def test_reuse_equals_own_prep_and_matches_oracle(kdkl, shape):
    T, d, V, K, chunk, tau, pad = shape
    w = WORKLOADS["small"].with_(T=T, d=d, V=V, K=K, chunk=chunk, tau=tau,
                                 seq_len=max(T // 3, 1), pad_frac=pad)
    x = make_inputs(w, seed=21)
    if x["mask"].sum() == 0:
        x["mask"][0] = 1
    l_own, dH_own, dW_own = _run(kdkl, x, tau, chunk, reuse=False, grad_loss=0.8)
    l_re, dH_re, dW_re = _run(kdkl, x, tau, chunk, reuse=True, grad_loss=0.8)
    assert l_own == l_re
    assert torch.equal(dH_own, dH_re) and torch.equal(dW_own, dW_re)
    H, W, idx, logit, mask = to_oracle(x)
    r_loss, _, _ = ok.forward(H, W, idx, logit, mask, tau)
    r_dH, r_dW = ok.backward(H, W, idx, logit, mask, tau, 0.8)
    assert abs(l_re - r_loss) <= LOSS_RTOL * abs(r_loss)
    assert rel_l2(dH_re.float().numpy(), r_dH) <= GRAD_REL_L2
    assert rel_l2(dW_re.numpy(), r_dW) <= GRAD_REL_L2


def test_reuse_with_another_chunk_and_edge_entries(kdkl):
    """The teacher rows do not depend on chunk: a backward with another chunk
    may reuse them. Repeated ids, -inf entries and a single-entry support go
    through the forward's sort."""
    w = WORKLOADS["small"].with_(T=96, d=64, V=500, K=12, chunk=32, tau=1.3)
    x = make_inputs(w, seed=11)
    lg, idx = x["topk_logit"], x["topk_idx"]
    lg[3, 5:] = float("-inf")
    idx[7, 4] = idx[7, 2]
    lg[9, 1:] = float("-inf")
    idx[40, :] = idx[40, 0]
    _, dH_a, dW_a = _run(kdkl, x, w.tau, 32, reuse=False, bwd_chunk=17)
    _, dH_b, dW_b = _run(kdkl, x, w.tau, 32, reuse=True, bwd_chunk=17)
    assert torch.equal(dH_a, dH_b) and torch.equal(dW_a, dW_b)
    H, W, i, l, m = to_oracle(x)
    r_dH, r_dW = ok.backward(H, W, i, l, m, w.tau, 1.0)
    assert rel_l2(dH_b.float().numpy(), r_dH) <= GRAD_REL_L2
    assert rel_l2(dW_b.numpy(), r_dW) <= GRAD_REL_L2


def test_reuse_of_the_mixed_forward(kdkl):
    w = WORKLOADS["small"].with_(T=150, d=64, V=1200, K=10, chunk=64, tau=1.5)
    x = make_inputs(w, seed=22)
    g = {k: v.cuda() for k, v in x.items()}
    labels = torch.randint(0, w.V, (w.T,), dtype=torch.int32,
                           generator=torch.Generator().manual_seed(3)).cuda()
    ws_f = torch.empty(kdkl.kd_kl_workspace_size(w.T, w.d, w.V, w.K, w.tau, w.chunk, 2),
                       dtype=torch.uint8, device="cuda")
    a = (g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], labels)
    kw = dict(temperature=w.tau, chunk=w.chunk, alpha=0.4, scale_tau_sq=True)
    _, lse, lse1, _ = kdkl.kd_kl_forward_ex(*a, workspace=ws_f, **kw)
    dH1, dW1 = kdkl.kd_kl_backward_ex(*a, lse, lse1, **kw)
    dH2, dW2 = kdkl.kd_kl_backward_ex(*a, lse, lse1, fwd_workspace=ws_f, **kw)
    torch.cuda.synchronize()
    assert torch.equal(dH1, dH2) and torch.equal(dW1, dW2)


def test_reuse_refused_for_another_problem(kdkl):
    w = WORKLOADS["small"].with_(T=64, d=32, V=300, K=4, chunk=16)
    x = make_inputs(w, seed=23)
    g = {k: v.cuda() for k, v in x.items()}
    ws_f = torch.empty(kdkl.kd_kl_workspace_size(64, 32, 300, 4, 1.0, 16, 0), dtype=torch.uint8,
                       device="cuda")
    _, lse, _ = kdkl.kd_kl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"],
                                   temperature=1.0, chunk=16, workspace=ws_f)
    with pytest.raises(kdkl.KDKLError) as e:  # another temperature: other teacher p
        kdkl.kd_kl_backward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], lse,
                            temperature=2.0, chunk=16, fwd_workspace=ws_f)
    assert e.value.code == 1
    with pytest.raises(kdkl.KDKLError) as e:  # a workspace no forward filled
        kdkl.kd_kl_backward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], lse,
                            temperature=1.0, chunk=16, fwd_workspace=torch.zeros_like(ws_f))
    assert e.value.code == 1


@pytest.mark.parametrize("K", [3, 16, 100, 256, 512])
def test_wide_and_packed_keys_agree(kdkl, K, monkeypatch):
    """Sort keys pack (id, position) into 32 bits when V * N < 2^32, else 64
    bits. Both orders are by id, then position, so the prepared rows, and all
    results, are the same bit for bit."""
    w = WORKLOADS["small"].with_(T=70, d=32, V=2 * K + 300, K=K, chunk=20, tau=1.1)
    x = make_inputs(w, seed=24)
    x["topk_idx"][5, 1] = x["topk_idx"][5, 0]  # a repeated id: order set by position
    runs = []
    for wide in ("0", "1"):
        monkeypatch.setenv("KDKL_PREP_WIDE", wide)
        g = {k: v.cuda() for k, v in x.items()}
        loss, lse, tkl = kdkl.kd_kl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"],
                                            g["mask"], temperature=w.tau, chunk=w.chunk,
                                            want_token_kl=True)
        dH, dW = kdkl.kd_kl_backward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"],
                                     lse, temperature=w.tau, chunk=w.chunk)
        torch.cuda.synchronize()
        runs.append([t.cpu() for t in (loss, lse, tkl, dH, dW)])
    for a, b in zip(*runs):
        assert torch.equal(a, b)
    H, W, i, l, m = to_oracle(x)
    r_loss, _, r_kl = ok.forward(H, W, i, l, m, w.tau)
    assert abs(runs[1][0].item() - r_loss) <= LOSS_RTOL * abs(r_loss)
    assert np.abs(runs[1][2].numpy() - r_kl).max() <= 1e-3 * max(1.0, np.abs(r_kl).max())
