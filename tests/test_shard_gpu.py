"""Token-sharded data parallelism through the CUDA library, on one GPU.

The loss is a mean over counted tokens, so a batch splits into token shards:
shard r computes its own loss_r over N_r counted tokens, the global loss is
sum_r N_r loss_r / sum_r N_r, and a backward called with grad_loss = N_r / N
gives shard r's part of the global gradients. dH rows are then final and dW
is the sum over shards. On several GPUs that sum is the ordinary data-parallel
all-reduce; here the shards run one after the other on one GPU and the sum is
taken by accumulate_dW into one dW. The combined results must match the
fp64 oracle on the whole batch, for the KL loss, the mixed soft + hard-label
loss and the reverse KL over the cached ids ("Making knowledge distillation
cheap enough to run at scale", section "Scaling to long contexts": the same
loss split over fewer or more GPUs)."""
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


def _case(seed, T=520, d=96, V=2600, K=12, tau=1.3, chunk=96):
    w = WORKLOADS["small"].with_(T=T, d=d, V=V, K=K, chunk=chunk, tau=tau, seq_len=130,
                                 pad_frac=0.3)
    x = make_inputs(w, seed=seed)
    labels = torch.randint(0, V, (T,), dtype=torch.int32,
                           generator=torch.Generator().manual_seed(seed))
    return w, x, labels


def _shards(T, bounds):
    return [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]


def _sharded(kdkl, w, x, labels, bounds, loss_kind):
    """Runs the shards through the library; returns (global loss, dH, dW)."""
    g = {k: v.cuda() for k, v in x.items()}
    lab = labels.cuda()
    mask = x["mask"]
    N = int(mask.sum())
    dW = torch.empty(w.V, w.d, dtype=torch.float32, device="cuda")
    dH_parts, num = [], 0.0
    for r, (lo, hi) in enumerate(_shards(w.T, bounds)):
        n_r = int(mask[lo:hi].sum())
        s = {k: v[lo:hi].contiguous() for k, v in g.items() if k != "W"}
        a = (s["H"], g["W"], s["topk_idx"], s["topk_logit"], s["mask"])
        kw = dict(temperature=w.tau, chunk=w.chunk)
        if loss_kind == "kl":
            loss, lse, _ = kdkl.kd_kl_forward(*a, **kw)
            dH, _ = kdkl.kd_kl_backward(*a, lse, grad_loss=n_r / N, dW=dW, accumulate_dW=r > 0,
                                        **kw)
        elif loss_kind == "mixed":
            lab_r = lab[lo:hi].contiguous()
            mk = dict(alpha=0.3, scale_tau_sq=True, **kw)
            loss, lse, lse1, _ = kdkl.kd_kl_forward_ex(*a, lab_r, **mk)
            dH, _ = kdkl.kd_kl_backward_ex(*a, lab_r, lse, lse1, grad_loss=n_r / N, dW=dW,
                                           accumulate_dW=r > 0, **mk)
        else:
            loss, _, gz = kdkl.kd_rkl_forward(*a, temperature=w.tau, want_grad_z=True)
            dH, _ = kdkl.kd_rkl_backward(*a, temperature=w.tau, grad_z=gz, grad_loss=n_r / N,
                                         dW=dW, accumulate_dW=r > 0)
        num += n_r * loss.item()
        dH_parts.append(dH)
    torch.cuda.synchronize()
    return num / N, torch.cat(dH_parts).float().cpu().numpy(), dW.cpu().numpy()


def _whole(w, x, labels, loss_kind):
    H, W, idx, logit, mask = to_oracle(x)
    lab = labels.numpy().astype(np.int64)
    if loss_kind == "kl":
        return (ok.forward(H, W, idx, logit, mask, w.tau)[0],
                *ok.backward(H, W, idx, logit, mask, w.tau, 1.0))
    if loss_kind == "mixed":
        return (ok.forward_mixed(H, W, idx, logit, mask, w.tau, 0.3, True, lab)[0],
                *ok.backward_mixed(H, W, idx, logit, mask, w.tau, 0.3, True, lab, 1.0))
    return (ok.reverse_kl_forward(H, W, idx, logit, mask, w.tau)[0],
            *ok.reverse_kl_backward(H, W, idx, logit, mask, w.tau, 1.0))


@pytest.mark.parametrize("loss_kind", ["kl", "mixed", "rkl"])
@pytest.mark.parametrize("bounds", [
    (0, 260, 520),        # two equal shards
    (0, 130, 333, 520),   # three unequal shards, cut inside sequences
    (0, 91, 130, 520),    # the middle shard is all padding (N_r = 0)
])
def test_shards_combine_to_the_whole_batch(kdkl, loss_kind, bounds):
    w, x, labels = _case(seed=31)
    if bounds == (0, 91, 130, 520):
        assert int(x["mask"][91:130].sum()) == 0  # the sequence tail padding
    loss, dH, dW = _sharded(kdkl, w, x, labels, bounds, loss_kind)
    r_loss, r_dH, r_dW = _whole(w, x, labels, loss_kind)
    assert abs(loss - r_loss) <= LOSS_RTOL * abs(r_loss), (loss, r_loss)
    assert rel_l2(dH, r_dH) <= GRAD_REL_L2
    assert rel_l2(dW, r_dW) <= GRAD_REL_L2
    assert not dH[x["mask"].numpy() == 0].any()  # masked rows exactly zero


def test_shards_at_the_bench_head_shape(kdkl):
    """Two token shards of 2048 tokens of the GPT-OSS-20B-like head
    (d = 2880, V = 201,088, K = 100) through the same sharded recipe. Only 40
    tokens, spread over both shards, are counted, so that the fp64 oracle can
    take them all within seconds: the loss, every row of dH, and dW on
    sampled vocabulary rows (half of them ids the teacher cache names)."""
    w = WORKLOADS["gptoss20b_32k"].with_(T=4096, teacher="uniform")
    x = make_inputs(w, seed=32)
    rng = np.random.default_rng(0)
    counted = np.sort(rng.choice(w.T, 40, replace=False))
    x["mask"].zero_()
    x["mask"][torch.from_numpy(counted)] = 1
    labels = torch.zeros(w.T, dtype=torch.int32)
    loss, dH, dW = _sharded(kdkl, w, x, labels, (0, 2048, 4096), "kl")
    H, W, idx, logit, _ = to_oracle(x)
    ones = np.ones(len(counted), dtype=np.uint8)
    Hc, ic, lc = H[counted], idx[counted], logit[counted]
    r_loss, _, _ = ok.forward(Hc, W, ic, lc, ones, w.tau)
    assert abs(loss - r_loss) <= LOSS_RTOL * abs(r_loss)
    G = ok.grad_logits(Hc, W, ic, lc, ones, w.tau, 1.0)
    assert rel_l2(dH[counted], G @ W) <= GRAD_REL_L2
    rest = np.setdiff1d(np.arange(w.T), counted)
    assert not dH[rest].any()
    vocab = np.unique(np.concatenate([rng.choice(ic.ravel(), 64, replace=False),
                                      rng.choice(w.V, 64, replace=False)]))
    assert rel_l2(dW[vocab], G[:, vocab].T @ Hc) <= GRAD_REL_L2
