"""Reverse KL over the cached ids on the GPU against the fp64 oracle: ragged
token counts, hidden sizes that leave lanes idle or span several 1024-column
passes, K above and below a warp, masked tokens, -inf teacher entries,
repeated ids, accumulation into dW, the degenerate cases, and the full-size
shapes (sparse mask, every touched dW row)."""
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


def _run(kdkl, x, tau, grad_loss=0.8, dW_init=None, use_grad_z=True):
    g = {k: v.cuda() for k, v in x.items()}
    loss, tok, gz = kdkl.kd_rkl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"],
                                        temperature=tau, want_token_rkl=True, want_grad_z=True)
    dW = None if dW_init is None else dW_init.cuda().clone()
    dH, dW = kdkl.kd_rkl_backward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"],
                                  temperature=tau, grad_z=gz if use_grad_z else None,
                                  grad_loss=grad_loss, dW=dW, accumulate_dW=dW_init is not None)
    torch.cuda.synchronize()
    return (loss.item(), tok.cpu().numpy().astype(np.float64),
            dH.float().cpu().numpy().astype(np.float64), dW.cpu().numpy().astype(np.float64),
            gz.cpu().numpy().astype(np.float64))


def _check(x, tau, got, grad_loss=0.8, dW_base=None):
    loss, tok, dH, dW, gz = got
    H, W, idx, logit, mask = to_oracle(x)
    r_loss, r_tok, _ = ok.reverse_kl_forward(H, W, idx, logit, mask, tau)
    r_gz = ok.reverse_kl_grad_z(H, W, idx, logit, mask, tau)
    r_dH, r_dW = ok.reverse_kl_backward(H, W, idx, logit, mask, tau, grad_loss)
    if dW_base is not None:
        r_dW = r_dW + dW_base
    assert abs(loss - r_loss) <= LOSS_RTOL * abs(r_loss) + 1e-6, (loss, r_loss)
    assert np.abs(tok - r_tok).max() <= 1e-3 * max(1.0, np.abs(r_tok).max())
    assert rel_l2(gz, r_gz) <= GRAD_REL_L2
    assert rel_l2(dH, r_dH) <= GRAD_REL_L2
    assert rel_l2(dW, r_dW) <= GRAD_REL_L2
    # masked tokens: no gradient at all
    assert np.all(dH[mask == 0] == 0.0) and np.all(gz[mask == 0] == 0.0)


@pytest.mark.parametrize("tau", [1.0, 2.0, 0.6])
@pytest.mark.parametrize("shape", [
    (131, 72, 1000, 7),      # ragged T, 9 of 32 lanes carry columns
    (300, 1160, 3000, 40),   # two 1024-column passes with a ragged tail, K > 32
    (64, 256, 500, 1),       # single-entry support: zero loss and zero gradient
    (517, 64, 300, 100),     # K close to V: ids repeat across tokens
])
def test_against_oracle(kdkl, tau, shape):
    T, d, V, K = shape
    w = WORKLOADS["small"].with_(T=T, d=d, V=V, K=K, tau=tau, seq_len=max(T // 3, 1),
                                 pad_frac=0.25)
    x = make_inputs(w, seed=21)
    got = _run(kdkl, x, tau)
    if K == 1:
        loss, tok, dH, dW, gz = got
        assert loss == 0.0 and np.all(tok == 0.0) and np.all(dH == 0.0) and np.all(dW == 0.0)
        assert np.all(gz == 0.0)
        return
    _check(x, tau, got)
    # the backward's own recompute of grad_z gives the same gradients
    again = _run(kdkl, x, tau, use_grad_z=False)
    assert np.array_equal(again[2], got[2]) and np.array_equal(again[3], got[3])


def test_neg_inf_entries_and_repeated_ids(kdkl):
    w = WORKLOADS["small"].with_(T=200, d=128, V=400, K=12, tau=1.3)
    x = make_inputs(w, seed=22)
    rng = np.random.default_rng(3)
    logit = x["topk_logit"].numpy()
    drop = rng.random(logit.shape) < 0.3
    drop[:, 0] = False  # every row keeps a finite entry
    logit[drop] = -np.inf
    idx = x["topk_idx"].numpy()
    idx[::5, 3] = idx[::5, 2]  # the same id twice in one row
    got = _run(kdkl, x, 1.3)
    _check(x, 1.3, got)


def test_accumulate_dW(kdkl):
    w = WORKLOADS["small"].with_(T=96, d=64, V=700, K=9, tau=1.0)
    x = make_inputs(w, seed=23)
    base = torch.from_numpy(np.random.default_rng(4).standard_normal((700, 64)).astype(np.float32))
    got = _run(kdkl, x, 1.0, grad_loss=1.7, dW_init=base)
    _check(x, 1.0, got, grad_loss=1.7, dW_base=base.numpy().astype(np.float64))


def test_matching_distributions_give_zero(kdkl):
    """Teacher logits equal to the student's own gathered logits (in fp32, up
    to a row constant): the loss and the gradient vanish to rounding."""
    w = WORKLOADS["small"].with_(T=128, d=256, V=1000, K=20, tau=1.0)
    x = make_inputs(w, seed=24)
    H, W, idx = x["H"].float(), x["W"].float(), x["topk_idx"].long()
    x["topk_logit"] = (torch.gather(H @ W.T, 1, idx) + 2.5).contiguous()
    loss, tok, dH, dW, _ = _run(kdkl, x, 1.0)
    assert abs(loss) < 1e-5 and np.abs(tok).max() < 1e-5
    assert np.abs(dH).max() < 1e-4 and np.abs(dW).max() < 1e-4


def test_all_masked_and_empty(kdkl):
    w = WORKLOADS["small"].with_(T=40, d=32, V=100, K=4)
    x = make_inputs(w, seed=25)
    x["mask"][:] = 0
    loss, tok, dH, dW, gz = _run(kdkl, x, 1.0)
    assert loss == 0.0 and np.all(dH == 0.0) and np.all(dW == 0.0)
    assert np.all(np.isfinite(tok)) and tok.max() > 0.0  # per-token values before masking
    assert np.all(gz == 0.0)
    H = torch.zeros((0, 32), dtype=torch.bfloat16, device="cuda")
    W = x["W"].cuda()
    idx = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    lg = torch.zeros((0, 4), dtype=torch.float32, device="cuda")
    loss, _, _ = kdkl.kd_rkl_forward(H, W, idx, lg)
    dH, dW = kdkl.kd_rkl_backward(H, W, idx, lg)
    torch.cuda.synchronize()
    assert loss.item() == 0.0 and dH.shape == (0, 32) and torch.count_nonzero(dW).item() == 0


def test_backward_is_bitwise_reproducible_and_heavy_ids(kdkl):
    """A few ids named by every token (buckets far longer than one dW segment)
    next to rare ones; two backward calls give identical bits."""
    w = WORKLOADS["small"].with_(T=1500, d=200, V=5000, K=24, tau=1.0, seq_len=500,
                                 pad_frac=0.1)
    x = make_inputs(w, seed=28)
    idx = x["topk_idx"].numpy()
    heavy = np.array([7, 4000, 4001], dtype=np.int32)
    for j, h in enumerate(heavy):  # keep rows duplicate-free: replace where absent
        col = idx[:, j]
        absent = ~(idx == h).any(axis=1)
        col[absent] = h
    got = _run(kdkl, x, 1.0)
    _check(x, 1.0, got)
    again = _run(kdkl, x, 1.0)
    assert np.array_equal(got[2], again[2]) and np.array_equal(got[3], again[3])


def test_index_out_of_range_is_reported(kdkl):
    w = WORKLOADS["small"].with_(T=64, d=16, V=100, K=3)
    x = make_inputs(w, seed=26)
    g = {k: v.cuda() for k, v in x.items()}
    g["topk_idx"][7, 1] = 100
    ws = torch.empty(kdkl.kd_rkl_workspace_size(64, 16, 100, 3), dtype=torch.uint8, device="cuda")
    kdkl.kd_rkl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], workspace=ws)
    assert kdkl.kd_kl_check_status(ws) == 4
    g["topk_idx"][7, 1] = -1
    kdkl.kd_rkl_backward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], workspace=ws)
    assert kdkl.kd_kl_check_status(ws) == 4
    g["topk_idx"][7, 1] = 5
    kdkl.kd_rkl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], workspace=ws)
    assert kdkl.kd_kl_check_status(ws) == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["gptoss20b_32k", "llama3b_8k", "padded_4x8k", "toyproj_256k"])
def test_full_size_sparse_mask(kdkl, name):
    """Full-size shapes. Only a sampled token set S counts (m = 0 elsewhere),
    so the oracle needs only the rows of S and the rows of W at their ids: it
    gives the exact loss, dH on S, and every dW row S touches; all other dW
    and dH rows must be exactly zero. Per-token values are checked on S."""
    w = WORKLOADS[name]
    x = make_inputs(w, seed=27, topk_device="cuda")
    T = w.T
    rng = np.random.default_rng(6)
    S = np.unique(np.concatenate([[0, 1, 127, T // 2, T - 2, T - 1],
                                  rng.choice(T, 90, replace=False)]))
    mask = torch.zeros(T, dtype=torch.uint8)
    mask[torch.from_numpy(S)] = 1
    g = {k: v.cuda() for k, v in x.items()}
    g["mask"] = mask.cuda()
    loss, tok, gz = kdkl.kd_rkl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"],
                                        g["mask"], temperature=w.tau, want_token_rkl=True,
                                        want_grad_z=True)
    dH, dW = kdkl.kd_rkl_backward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"],
                                  temperature=w.tau, grad_z=gz, grad_loss=1.0)
    torch.cuda.synchronize()
    idx_S = x["topk_idx"].numpy()[S].astype(np.int64)
    touched, local = np.unique(idx_S, return_inverse=True)
    local = local.reshape(idx_S.shape)
    H_S = ok.bf16_bits_to_f64(x["H"][torch.from_numpy(S)].view(torch.int16).numpy())
    W_T = ok.bf16_bits_to_f64(x["W"][torch.from_numpy(touched)].view(torch.int16).numpy())
    logit_S = x["topk_logit"].numpy()[S].astype(np.float64)
    ones = np.ones(len(S), dtype=np.uint8)
    r_loss, r_tok, _ = ok.reverse_kl_forward(H_S, W_T, local, logit_S, ones, w.tau)
    r_dH, r_dW = ok.reverse_kl_backward(H_S, W_T, local, logit_S, ones, w.tau, 1.0)
    assert abs(loss.item() - r_loss) <= LOSS_RTOL * abs(r_loss)
    tok_S = tok[torch.from_numpy(S).cuda()].cpu().numpy().astype(np.float64)
    assert np.abs(tok_S - r_tok).max() <= 1e-3 * max(1.0, np.abs(r_tok).max())
    s_dev = torch.from_numpy(S).cuda()
    assert rel_l2(dH[s_dev].float().cpu().numpy(), r_dH) <= GRAD_REL_L2
    t_dev = torch.from_numpy(touched).cuda()
    assert rel_l2(dW[t_dev].cpu().numpy(), r_dW) <= GRAD_REL_L2
    # everything outside S (tokens) and outside the touched ids (vocabulary) is zero
    keep_rows = torch.zeros(T, dtype=torch.bool, device="cuda")
    keep_rows[s_dev] = True
    assert torch.count_nonzero(dH[~keep_rows]).item() == 0
    keep_v = torch.zeros(w.V, dtype=torch.bool, device="cuda")
    keep_v[t_dev] = True
    assert torch.count_nonzero(dW[~keep_v]).item() == 0


def test_null_mask_equals_all_ones(kdkl):
    """mask = NULL counts every token: the same bits as an all-ones mask."""
    w = WORKLOADS["small"].with_(T=150, d=96, V=900, K=11, tau=1.2)
    x = make_inputs(w, seed=29)
    g = {k: v.cuda() for k, v in x.items()}
    ones = torch.ones(w.T, dtype=torch.uint8, device="cuda")
    out = []
    for m in (None, ones):
        loss, tok, gz = kdkl.kd_rkl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], m,
                                            temperature=w.tau, want_token_rkl=True,
                                            want_grad_z=True)
        dH, dW = kdkl.kd_rkl_backward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], m,
                                      temperature=w.tau, grad_z=gz)
        out.append((loss, tok, gz, dH, dW))
    torch.cuda.synchronize()
    for a, b in zip(*out):
        assert torch.equal(a, b)
