"""The loss calls inside a CUDA graph. Forward + backward of the KL path (and of
the reverse-KL variant) are captured once on torch's graph stream and
replayed. Every reduction runs in a fixed order, so a replay must equal the
eager calls bit for bit; after new inputs are copied into the captured
buffers, a replay must equal eager calls on those new inputs."""
import numpy as np
import pytest
import torch

from lm_head_top_gb300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

SHAPE = dict(T=384, d=320, V=3000, K=20, chunk=128, tau=1.5, seq_len=128, pad_frac=0.2)


@pytest.fixture(scope="module")
def kdkl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_top_gb300 import kdkl as m
    m.load()
    return m


def _inputs(seed):
    w = WORKLOADS["small"].with_(**SHAPE)
    return w, {k: v.cuda() for k, v in make_inputs(w, seed=seed).items()}


class KLStep:
    """Static buffers for one fused KL forward + backward."""

    def __init__(self, kdkl, w, x):
        self.kdkl, self.w = kdkl, w
        self.x = {k: v.clone() for k, v in x.items()}
        T, d, V, K = w.T, w.d, w.V, w.K
        dev = x["H"].device
        self.ws_f = torch.empty(kdkl.kd_kl_workspace_size(T, d, V, K, w.tau, w.chunk, 0),
                                dtype=torch.uint8, device=dev)
        self.ws_b = torch.empty(kdkl.kd_kl_workspace_size(T, d, V, K, w.tau, w.chunk, 1),
                                dtype=torch.uint8, device=dev)
        self.loss = torch.empty(1, device=dev)
        self.lse = torch.empty(T, device=dev)
        self.tok = torch.empty(T, device=dev)
        self.dH = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty(V, d, device=dev)

    def __call__(self):
        k, w, x = self.kdkl, self.w, self.x
        k.kd_kl_forward(x["H"], x["W"], x["topk_idx"], x["topk_logit"], x["mask"],
                        temperature=w.tau, chunk=w.chunk, loss=self.loss, lse=self.lse,
                        token_kl=self.tok, workspace=self.ws_f)
        k.kd_kl_backward(x["H"], x["W"], x["topk_idx"], x["topk_logit"], x["mask"], self.lse,
                         temperature=w.tau, chunk=w.chunk, grad_loss=0.5, dH=self.dH, dW=self.dW,
                         workspace=self.ws_b)

    def outputs(self):
        return [t.clone() for t in (self.loss, self.lse, self.tok, self.dH, self.dW)]


class RKLStep:
    """Static buffers for one reverse-KL forward + backward (saved dloss/dz)."""

    def __init__(self, kdkl, w, x):
        self.kdkl, self.w = kdkl, w
        self.x = {k: v.clone() for k, v in x.items()}
        T, d, V, K = w.T, w.d, w.V, w.K
        dev = x["H"].device
        self.ws = torch.empty(kdkl.kd_rkl_workspace_size(T, d, V, K, w.tau), dtype=torch.uint8,
                              device=dev)
        self.loss = torch.empty(1, device=dev)
        self.tok = torch.empty(T, device=dev)
        self.gz = torch.empty(T, K, device=dev)
        self.dH = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty(V, d, device=dev)

    def __call__(self):
        k, w, x = self.kdkl, self.w, self.x
        k.kd_rkl_forward(x["H"], x["W"], x["topk_idx"], x["topk_logit"], x["mask"],
                         temperature=w.tau, loss=self.loss, token_rkl=self.tok, grad_z=self.gz,
                         workspace=self.ws)
        k.kd_rkl_backward(x["H"], x["W"], x["topk_idx"], x["topk_logit"], x["mask"],
                          temperature=w.tau, grad_z=self.gz, grad_loss=0.5, dH=self.dH,
                          dW=self.dW, workspace=self.ws)

    def outputs(self):
        return [t.clone() for t in (self.loss, self.tok, self.gz, self.dH, self.dW)]


def _eager(cls, kdkl, w, x):
    step = cls(kdkl, w, x)
    step()
    torch.cuda.synchronize()
    return step.outputs()


@pytest.mark.parametrize("cls", [KLStep, RKLStep], ids=["kl", "rkl"])
def test_graph_replay_matches_eager(kdkl, cls):
    w, x1 = _inputs(31)
    _, x2 = _inputs(32)
    want1 = _eager(cls, kdkl, w, x1)
    want2 = _eager(cls, kdkl, w, x2)

    step = cls(kdkl, w, x1)
    step()  # first call on this device outside the capture (attribute and driver lookups)
    torch.cuda.synchronize()
    n0 = kdkl.kd_launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    per_step = kdkl.kd_launch_count() - n0
    assert per_step > 0

    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    # replays launch nothing through the library's host path
    assert kdkl.kd_launch_count() - n0 == per_step
    for got, want in zip(step.outputs(), want1):
        assert torch.equal(got, want)

    for k in step.x:  # new inputs into the captured buffers
        step.x[k].copy_(x2[k])
    graph.replay()
    torch.cuda.synchronize()
    for got, want in zip(step.outputs(), want2):
        assert torch.equal(got, want)
    assert not np.isclose(want1[0].item(), want2[0].item())
