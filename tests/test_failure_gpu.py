"""Failure detection on the GPU without a fault: a stall injected on purpose
(the producer warp issues nothing, so nothing ever completes the MMA warp's
first wait) must end in KD_ERR_TIMEOUT after the short injected wait limit.
The kernel unwinds (drains, frees TMEM) and the context stays usable."""
import numpy as np
import pytest
import torch

from lm_head_top_gb300.inputs import WORKLOADS, make_inputs
from tests._helpers import run_gpu, to_oracle
import oracle.kl_oracle as ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kdkl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_top_gb300 import kdkl as m
    m.load()
    return m


def test_injected_stall_times_out_and_context_survives(kdkl, monkeypatch):
    w = WORKLOADS["small"].with_(T=300, d=64, V=1100, K=6, chunk=128)
    x = make_inputs(w, seed=3)
    g = {k: v.cuda() for k, v in x.items()}
    ws_f = torch.empty(kdkl.kd_kl_workspace_size(w.T, w.d, w.V, w.K, 1.0, w.chunk, 0),
                       dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(kdkl.kd_kl_workspace_size(w.T, w.d, w.V, w.K, 1.0, w.chunk, 1),
                       dtype=torch.uint8, device="cuda")

    monkeypatch.setenv("KDKL_INJECT_STALL", "1")
    _, lse, _ = kdkl.kd_kl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"],
                                   chunk=w.chunk, workspace=ws_f)
    assert kdkl.kd_kl_check_status(ws_f) == 7  # KD_ERR_TIMEOUT
    kdkl.kd_kl_backward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], lse,
                        chunk=w.chunk, workspace=ws_b)
    assert kdkl.kd_kl_check_status(ws_b) == 7
    monkeypatch.delenv("KDKL_INJECT_STALL")

    # same process, same context: a normal call is correct again
    kdkl.kd_kl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"],
                       chunk=w.chunk, workspace=ws_f)
    assert kdkl.kd_kl_check_status(ws_f) == 0
    out = run_gpu(kdkl, x, 1.0, w.chunk)
    H, W, idx, logit, mask = to_oracle(x)
    r_loss = ok.forward(H, W, idx, logit, mask, 1.0)[0]
    assert abs(out["loss"] - r_loss) <= 1e-3 * abs(r_loss)
    assert np.isfinite(out["dW"]).all()
