"""kd_kl_forward_noalloc: the forward for callers that cannot allocate device
memory (code inside a host framework whose memory pool owns the GPU's free
memory, or a loop that must not risk a device-synchronising cudaMalloc). It
must give the results of kd_kl_forward with a caller-provided workspace, and
of the fp64 oracle, call after call; allocate nothing; report device-detected
errors through kd_kl_noalloc_check_status; and refuse problems larger than its
fixed scratch array.

Collected last on purpose (file name), so a stop-at-first-failure run has
already run every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle.kl_oracle as ok
from lm_head_top_gb300.inputs import WORKLOADS, make_inputs
from tests._helpers import LOSS_RTOL, LSE_ATOL, max_err_counted, to_oracle

pytestmark = pytest.mark.gpu

KD_ERR_INDEX_RANGE = 4
KD_ERR_WORKSPACE = 5


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_top_gb300 import kdkl
    return kdkl, kdkl.load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(L, p, g, out):
    return L.kd_kl_forward_noalloc(ctypes.byref(p), _ptr(g["H"]), _ptr(g["W"]),
                                   _ptr(g["topk_idx"]), _ptr(g["topk_logit"]), _ptr(g["mask"]),
                                   _ptr(out["loss"]), _ptr(out["lse"]), _ptr(out["kl"]),
                                   _stream())


def _call_both(kdkl, L, x, w):
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in x.items()}
    T = w.T
    p = kdkl.kd_kl_problem(w.T, w.d, w.V, w.K, w.tau, w.chunk)

    # the existing entry point, with a workspace the caller allocates
    ws = torch.empty(L.kd_kl_workspace_size(ctypes.byref(p), 0), dtype=torch.uint8, device=dev)
    ref = {"loss": torch.empty(1, device=dev), "lse": torch.empty(T, device=dev),
           "kl": torch.empty(T, device=dev)}
    rc = L.kd_kl_forward(ctypes.byref(p), _ptr(g["H"]), _ptr(g["W"]), _ptr(g["topk_idx"]),
                         _ptr(g["topk_logit"]), _ptr(g["mask"]), _ptr(ref["loss"]),
                         _ptr(ref["lse"]), _ptr(ref["kl"]), _ptr(ws), ws.numel(), _stream())
    assert rc == 0

    # the allocation-free entry point; outputs are poisoned first
    out = {k: torch.full_like(v, float("nan")) for k, v in ref.items()}
    rc = _noalloc(L, p, g, out)
    assert rc == 0, kdkl.kd_status_string(rc)
    assert L.kd_kl_noalloc_check_status(_stream()) == 0
    torch.cuda.synchronize(dev)
    return ({k: v.cpu().numpy().astype(np.float64) for k, v in ref.items()},
            {k: v.cpu().numpy().astype(np.float64) for k, v in out.items()})


def test_matches_existing_forward_and_oracle_on_consecutive_calls(lib):
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
        # and against the oracle, independently of the other entry point
        H, W, idx, logit, mask = to_oracle(x)
        r_loss, r_lse, r_kl = ok.forward(H, W, idx, logit, mask, w.tau)
        assert abs(out["loss"][0] - r_loss) <= LOSS_RTOL * abs(r_loss)
        assert max_err_counted(out["lse"], r_lse, mask) <= LSE_ATOL
        assert max_err_counted(out["kl"], r_kl, mask) <= 1e-3 * max(1.0, np.abs(r_kl).max())


def test_allocates_nothing(lib):
    """After a first call on the device (its one-time set-up), further calls
    leave torch's allocated bytes and the device's free bytes unchanged."""
    kdkl, L = lib
    w = WORKLOADS["small"].with_(T=600, d=128, V=4000, K=16, chunk=64, tau=1.0)
    x = make_inputs(w, seed=14)
    g = {k: v.cuda() for k, v in x.items()}
    p = kdkl.kd_kl_problem(w.T, w.d, w.V, w.K, w.tau, w.chunk)
    out = {"loss": torch.empty(1, device="cuda"), "lse": torch.empty(w.T, device="cuda"),
           "kl": torch.empty(w.T, device="cuda")}
    assert _noalloc(L, p, g, out) == 0
    torch.cuda.synchronize()
    first = out["loss"].item()
    alloc0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _noalloc(L, p, g, out) == 0
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    assert out["loss"].item() == first  # the same inputs give the same bits


def test_device_detected_errors_are_read_back(lib):
    """An id outside [0, V) is recorded in the scratch array's status word and
    read with kd_kl_noalloc_check_status; the next clean call clears it."""
    kdkl, L = lib
    w = WORKLOADS["small"].with_(T=64, d=16, V=100, K=3, chunk=16)
    x = make_inputs(w, seed=7)
    x["topk_idx"][5, 1] = 100  # == V
    g = {k: v.cuda() for k, v in x.items()}
    p = kdkl.kd_kl_problem(w.T, w.d, w.V, w.K, w.tau, w.chunk)
    out = {"loss": torch.empty(1, device="cuda"), "lse": torch.empty(w.T, device="cuda"),
           "kl": None}
    assert _noalloc(L, p, g, out) == 0
    assert L.kd_kl_noalloc_check_status(_stream()) == KD_ERR_INDEX_RANGE
    x["topk_idx"][5, 1] = 3
    g = {k: v.cuda() for k, v in x.items()}
    assert _noalloc(L, p, g, out) == 0
    assert L.kd_kl_noalloc_check_status(_stream()) == 0


def test_rejects_problems_beyond_the_scratch_array(lib):
    kdkl, L = lib
    dev = torch.device("cuda:0")
    # 32768 tokens x 512 teacher entries need 128 MiB of sorted (id, p) alone
    p = kdkl.kd_kl_problem(32768, 64, 4096, 512, 1.0, 1024)
    assert L.kd_kl_workspace_size(ctypes.byref(p), 0) > (64 << 20)
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device=dev)  # never read: rejected first
    rc = L.kd_kl_forward_noalloc(ctypes.byref(p), _ptr(buf), _ptr(buf), _ptr(buf), _ptr(buf), None,
                                 _ptr(buf), _ptr(buf), None, _stream())
    assert rc == KD_ERR_WORKSPACE
