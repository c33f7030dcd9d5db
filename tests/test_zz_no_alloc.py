"""kd_kl_forward_noalloc: the forward for callers that cannot allocate device
memory (a host framework whose pool owns the GPU's free memory, or a loop that
must not risk a device-synchronising cudaMalloc). It must give the same
results as kd_kl_forward with a caller-provided workspace, call after call,
and refuse problems larger than its fixed scratch array.

Collected last on purpose (file name), so a stop-at-first-failure run has
already run every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from lm_head_top_gb300.inputs import WORKLOADS, make_inputs
from tests._helpers import LOSS_RTOL, LSE_ATOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_top_gb300 import kdkl
    return kdkl, kdkl.load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_both(kdkl, lib, x, w):
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in x.items()}
    T = w.T
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    p = kdkl.kd_kl_problem(w.T, w.d, w.V, w.K, w.tau, w.chunk)

    # the existing entry point, with a workspace the caller allocates
    ws = torch.empty(lib.kd_kl_workspace_size(ctypes.byref(p), 0), dtype=torch.uint8, device=dev)
    ref = {"loss": torch.empty(1, device=dev), "lse": torch.empty(T, device=dev),
           "kl": torch.empty(T, device=dev)}
    rc = lib.kd_kl_forward(ctypes.byref(p), _ptr(g["H"]), _ptr(g["W"]), _ptr(g["topk_idx"]),
                           _ptr(g["topk_logit"]), _ptr(g["mask"]), _ptr(ref["loss"]),
                           _ptr(ref["lse"]), _ptr(ref["kl"]), _ptr(ws), ws.numel(), stream)
    assert rc == 0

    # the allocation-free entry point; outputs are poisoned first
    out = {k: torch.full_like(v, float("nan")) for k, v in ref.items()}
    rc = lib.kd_kl_forward_noalloc(ctypes.byref(p), _ptr(g["H"]), _ptr(g["W"]),
                                   _ptr(g["topk_idx"]), _ptr(g["topk_logit"]), _ptr(g["mask"]),
                                   _ptr(out["loss"]), _ptr(out["lse"]), _ptr(out["kl"]), stream)
    assert rc == 0, kdkl.kd_status_string(rc)
    torch.cuda.synchronize(dev)
    return ({k: v.cpu().numpy().astype(np.float64) for k, v in ref.items()},
            {k: v.cpu().numpy().astype(np.float64) for k, v in out.items()})


def test_matches_existing_forward_on_consecutive_calls(lib):
    kdkl, L = lib
    cases = [
        WORKLOADS["small"].with_(T=1000, d=192, V=5000, K=24, chunk=64, tau=1.0),
        # second call: different sizes, temperature and a padded mask, so any
        # state left in the shared scratch by the first call would show
        WORKLOADS["small"].with_(T=777, d=136, V=3100, K=9, chunk=50, tau=2.0, seq_len=259,
                                 pad_frac=0.3),
    ]
    for i, w in enumerate(cases):
        x = make_inputs(w, seed=10 + i)
        ref, out = _call_both(kdkl, L, x, w)
        assert abs(out["loss"][0] - ref["loss"][0]) <= LOSS_RTOL * abs(ref["loss"][0])
        assert np.abs(out["lse"] - ref["lse"]).max() <= LSE_ATOL
        assert np.abs(out["kl"] - ref["kl"]).max() <= 1e-3 * max(1.0, np.abs(ref["kl"]).max())


def test_rejects_problems_beyond_the_scratch_array(lib):
    kdkl, L = lib
    dev = torch.device("cuda:0")
    # 32768 tokens x 512 teacher entries need 128 MiB of sorted (id, p) alone
    p = kdkl.kd_kl_problem(32768, 64, 4096, 512, 1.0, 1024)
    assert L.kd_kl_workspace_size(ctypes.byref(p), 0) > (64 << 20)
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device=dev)  # never read: rejected first
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = L.kd_kl_forward_noalloc(ctypes.byref(p), _ptr(buf), _ptr(buf), _ptr(buf), _ptr(buf), None,
                                 _ptr(buf), _ptr(buf), None, stream)
    assert rc == 5  # KD_ERR_WORKSPACE
