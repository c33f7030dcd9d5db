"""CUDA path (through the C ABI) against the fp64 oracle, element by element,
on identical seeded inputs. Sizes here finish in the oracle within seconds and
still span several 128 x 256 tiles, vocabulary slabs / token chunks and
ragged tails."""
import numpy as np
import pytest
import torch

import oracle.kl_oracle as ok
from lm_head_top_gb300.inputs import WORKLOADS, make_inputs
from tests._helpers import (GRAD_REL_L2, LOSS_RTOL, LSE_ATOL, max_err_counted, rel_l2, run_gpu,
                            to_oracle)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kdkl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_top_gb300 import kdkl as m
    m.load()
    return m


def _compare(out, x, tau, grad_loss=1.0, dW_init=None):
    H, W, idx, logit, mask = to_oracle(x)
    r_loss, r_lse, r_kl = ok.forward(H, W, idx, logit, mask, tau)
    r_dH, r_dW = ok.backward(H, W, idx, logit, mask, tau, grad_loss)
    if dW_init is not None:
        r_dW = r_dW + dW_init.numpy().astype(np.float64)
    keep = mask != 0
    errs = {
        "loss": abs(out["loss"] - r_loss) / max(abs(r_loss), 1e-30),
        # per-token outputs on counted tokens (masked ones read 0)
        "lse": max_err_counted(out["lse"], r_lse, mask),
        "kl": max_err_counted(out["token_kl"], r_kl, mask),
        "dH": rel_l2(out["dH"], r_dH),
        "dW": rel_l2(out["dW"], r_dW),
    }
    assert errs["loss"] <= LOSS_RTOL, errs
    assert errs["lse"] <= LSE_ATOL, errs
    assert errs["kl"] <= 1e-3 * max(1.0, float(np.abs(r_kl).max())), errs
    assert errs["dH"] <= GRAD_REL_L2, errs
    assert errs["dW"] <= GRAD_REL_L2, errs
    # masked rows of dH are exactly zero
    assert not out["dH"][~keep].any()
    return errs


def test_small_workload(kdkl):
    w = WORKLOADS["small"]
    x = make_inputs(w, seed=0)
    _compare(run_gpu(kdkl, x, w.tau, w.chunk), x, w.tau)


@pytest.mark.parametrize("shape", [
    # T, d, V, K, chunk, tau : ragged in every dimension, several vocabulary slabs
    (131, 72, 1000, 7, 50, 2.0),
    # more tokens than vocabulary: token chunks (dW accumulated across chunks)
    (700, 64, 300, 5, 200, 1.0),
    # one token, one teacher entry
    (1, 8, 40, 1, 1, 1.0),
    # K = V: the teacher covers the whole vocabulary
    (64, 32, 48, 48, 16, 0.5),
    # K = 512 (largest), V just above
    (40, 48, 600, 512, 7, 1.0),
    # hidden sizes whose last 256-wide dH / dW column tile is at most half
    # full: that tile runs 128 wide
    (200, 576, 900, 10, 70, 1.0),
    (129, 384, 777, 3, 129, 1.5),
    # last column tile more than half full: it stays 256 wide
    (150, 448, 900, 10, 70, 1.0),
])
def test_ragged_shapes(kdkl, shape):
    T, d, V, K, chunk, tau = shape
    w = WORKLOADS["small"].with_(T=T, d=d, V=V, K=K, chunk=chunk, tau=tau,
                                 seq_len=max(T // 3, 1), pad_frac=0.25)
    x = make_inputs(w, seed=1)
    if x["mask"].sum() == 0:
        x["mask"][0] = 1
    _compare(run_gpu(kdkl, x, tau, chunk, grad_loss=0.75), x, tau, grad_loss=0.75)


def test_accumulate_dW(kdkl):
    w = WORKLOADS["small"].with_(T=300, d=64, V=2000, K=9, chunk=100)
    x = make_inputs(w, seed=2)
    dW0 = torch.randn(2000, 64, dtype=torch.float32) * 1e-3
    _compare(run_gpu(kdkl, x, w.tau, w.chunk, dW_init=dW0), x, w.tau, dW_init=dW0)


def test_half_overlap_teacher(kdkl):
    w = WORKLOADS["small"].with_(T=384, d=128, V=3000, K=20, chunk=128, teacher="half_overlap")
    x = make_inputs(w, seed=3, topk_device="cpu")
    _compare(run_gpu(kdkl, x, w.tau, w.chunk), x, w.tau)


def test_chunk_invariance(kdkl):
    w = WORKLOADS["small"].with_(T=256, d=64, V=2500, K=10)
    x = make_inputs(w, seed=4)
    outs = [run_gpu(kdkl, x, 1.0, c) for c in (1, 37, 256, 100000)]
    for o in outs[1:]:
        assert o["loss"] == outs[0]["loss"]  # the forward does not depend on chunk
        assert rel_l2(o["dH"], outs[0]["dH"]) < 1e-2
        assert rel_l2(o["dW"], outs[0]["dW"]) < 1e-5


def test_all_masked(kdkl):
    w = WORKLOADS["small"].with_(T=130, d=32, V=700, K=4, chunk=64)
    x = make_inputs(w, seed=5)
    x["mask"].zero_()
    out = run_gpu(kdkl, x, 1.0, 64)
    assert out["loss"] == 0.0
    assert not out["dH"].any() and not out["dW"].any()


def test_no_mask_pointer_means_all_tokens(kdkl):
    w = WORKLOADS["small"].with_(T=200, d=40, V=900, K=6, chunk=64)
    x = make_inputs(w, seed=6)
    a = run_gpu(kdkl, x, 1.0, 64, mask=False)
    b = run_gpu(kdkl, x, 1.0, 64, mask=True)
    assert a["loss"] == b["loss"]
    assert rel_l2(a["dW"], b["dW"]) < 1e-6


def test_zero_tokens(kdkl):
    dev = "cuda:0"
    H = torch.empty(0, 16, dtype=torch.bfloat16, device=dev)
    W = torch.randn(50, 16, device=dev).to(torch.bfloat16)
    idx = torch.empty(0, 3, dtype=torch.int32, device=dev)
    lg = torch.empty(0, 3, dtype=torch.float32, device=dev)
    loss, lse, _ = kdkl.kd_kl_forward(H, W, idx, lg, None, temperature=1.0, chunk=8)
    dH, dW = kdkl.kd_kl_backward(H, W, idx, lg, None, lse, temperature=1.0, chunk=8)
    torch.cuda.synchronize()
    assert loss.item() == 0.0 and dW.abs().max().item() == 0.0


def test_device_detected_index_error(kdkl):
    w = WORKLOADS["small"].with_(T=64, d=16, V=100, K=3, chunk=16)
    x = make_inputs(w, seed=7)
    x["topk_idx"][5, 1] = 100  # == V: out of range
    g = {k: v.cuda() for k, v in x.items()}
    ws = torch.empty(kdkl.kd_kl_workspace_size(64, 16, 100, 3, 1.0, 16, 0), dtype=torch.uint8,
                     device="cuda")
    kdkl.kd_kl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], chunk=16,
                       workspace=ws)
    assert kdkl.kd_kl_check_status(ws) == 4  # KD_ERR_INDEX_RANGE
    x["topk_idx"][5, 1] = 3
    g = {k: v.cuda() for k, v in x.items()}
    kdkl.kd_kl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], chunk=16,
                       workspace=ws)
    assert kdkl.kd_kl_check_status(ws) == 0


def test_timing_and_launch_count(kdkl):
    w = WORKLOADS["small"].with_(T=128, d=64, V=1024, K=8, chunk=64)
    x = make_inputs(w, seed=8)
    before = kdkl.kd_launch_count()
    kdkl.kd_timing_begin()
    run_gpu(kdkl, x, 1.0, 64)
    rows = kdkl.kd_timing_end()
    names = {r[0] for r in rows}
    assert {"teacher_prep", "fwd_lse_gemm", "lse_combine", "loss_finalize", "bwd_grad_gemm",
            "dW_dH_gemm", "f32_to_bf16", "mask_scan", "gather_rows"} <= names
    assert kdkl.kd_launch_count() - before == sum(r[1] for r in rows)
    assert all(r[2] > 0 for r in rows)


def test_teacher_edge_entries(kdkl):
    """-inf teacher logits (p = 0, outside the support), ids repeated within a
    row (entries add: reading 6) and a row whose support is one entry, across
    several token chunks and vocabulary slabs."""
    w = WORKLOADS["small"].with_(T=96, d=64, V=500, K=12, chunk=32, tau=1.3)
    x = make_inputs(w, seed=11)
    lg, idx = x["topk_logit"], x["topk_idx"]
    lg[3, 5:] = float("-inf")            # half the row outside the support
    idx[7, 4] = idx[7, 2]                # a repeated id
    lg[9, 1:] = float("-inf")            # a single-entry support
    idx[11, 1] = idx[11, 0]              # repeat, and the repeat dropped
    lg[11, 1] = float("-inf")
    idx[40, :] = idx[40, 0]              # one id named K times
    _compare(run_gpu(kdkl, x, w.tau, w.chunk, grad_loss=0.5), x, w.tau, grad_loss=0.5)


def test_large_logits(kdkl):
    """Logits of a few hundred at a sharp temperature: the online
    logsumexp must not overflow, and the loss stays exact."""
    w = WORKLOADS["small"].with_(T=160, d=96, V=1500, K=16, chunk=64, tau=0.5)
    x = make_inputs(w, seed=12)
    x["H"] = (x["H"].float() * 60.0).to(torch.bfloat16)   # z ~ N(0, 60^2)
    x["topk_logit"] = x["topk_logit"] * 40.0
    out = run_gpu(kdkl, x, w.tau, w.chunk)
    assert np.isfinite(out["loss"]) and np.isfinite(out["lse"]).all()
    _compare(out, x, w.tau)


@pytest.mark.parametrize("bad", ["all_neg_inf", "nan", "pos_inf"])
def test_unusable_teacher_row_is_reported(kdkl, bad):
    """A teacher row with no finite logit, a NaN or +inf is an invalid input:
    the device status says KD_ERR_INVALID_ARG (1); a clean call afterwards on
    the same workspace reports 0."""
    w = WORKLOADS["small"].with_(T=64, d=16, V=100, K=3, chunk=16)
    x = make_inputs(w, seed=13)
    row = x["topk_logit"][9]
    if bad == "all_neg_inf":
        row[:] = float("-inf")
    elif bad == "nan":
        row[1] = float("nan")
    else:
        row[0] = float("inf")
    g = {k: v.cuda() for k, v in x.items()}
    ws = torch.empty(kdkl.kd_kl_workspace_size(64, 16, 100, 3, 1.0, 16, 0), dtype=torch.uint8,
                     device="cuda")
    kdkl.kd_kl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], chunk=16,
                       workspace=ws)
    assert kdkl.kd_kl_check_status(ws) == 1
    clean = make_inputs(w, seed=13)
    g = {k: v.cuda() for k, v in clean.items()}
    kdkl.kd_kl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], chunk=16,
                       workspace=ws)
    assert kdkl.kd_kl_check_status(ws) == 0


def test_mask_compaction_across_scan_tiles(kdkl):
    """A mask with scattered and long runs of masked tokens over 70,000 tokens
    (the compaction scan takes 32,768 tokens per pass: two full passes and a
    partial one). Counted tokens must match the oracle, masked ones read 0,
    and masked dH rows are exact zeros."""
    w = WORKLOADS["small"].with_(T=70000, d=64, V=520, K=8, chunk=4096, tau=1.2)
    x = make_inputs(w, seed=41)
    rng = np.random.default_rng(41)
    m = (rng.random(w.T) < 0.7).astype(np.uint8)   # scattered
    m[10000:20000] = 0                             # a run across no tile edge
    m[32700:32900] = 0                             # a run across the first tile edge
    m[65530:65540] = 1                             # counted tokens around the second edge
    x["mask"] = torch.from_numpy(m)
    _compare(run_gpu(kdkl, x, w.tau, w.chunk), x, w.tau)


@pytest.mark.parametrize("shape", [
    # T, d, V, K, chunk : d = 2880 is 11 column tiles of 256 and one of 64
    (512, 2880, 5000, 32, 2048),
    (300, 320, 5000, 8, 1000),
    (64, 72, 900, 4, 300),
])
def test_narrow_last_column_tile(kdkl, shape, monkeypatch):
    """The last dH / dW column tile, when at most half full, multiplies
    N = 128 instead of 256 and copies half the B rows. Each output element
    still sums the same products in the same k order, so dH and dW equal
    those of the full-width tile bit for bit, and both match the oracle."""
    T, d, V, K, chunk = shape
    w = WORKLOADS["small"].with_(T=T, d=d, V=V, K=K, chunk=chunk, tau=1.0,
                                 seq_len=max(T // 4, 1), pad_frac=0.1)
    x = make_inputs(w, seed=31)
    runs = {}
    for narrow in ("0", "1"):
        monkeypatch.setenv("KDKL_NARROW_LAST", narrow)
        runs[narrow] = run_gpu(kdkl, x, w.tau, w.chunk, grad_loss=0.5)
    for key in ("dH", "dW"):
        assert np.array_equal(runs["0"][key], runs["1"][key]), key
    _compare(runs["1"], x, w.tau, grad_loss=0.5)


@pytest.mark.parametrize("shape", [
    # T, d, V, K, chunk: vocabulary slabs whose dW and dH jobs are a few waves
    (700, 320, 9000, 16, 300),
    (200, 72, 3000, 8, 100),
])
def test_dual_and_separate_dh_dw_launches_agree(kdkl, shape, monkeypatch):
    """dW and dH of a block run as one launch (both jobs' units in one
    sequence) or as two; each output element sums the same products in the
    same order either way, so the two give the same bits, and the oracle's
    results."""
    T, d, V, K, chunk = shape
    w = WORKLOADS["small"].with_(T=T, d=d, V=V, K=K, chunk=chunk, tau=1.3,
                                 seq_len=max(T // 4, 1), pad_frac=0.15)
    x = make_inputs(w, seed=33)
    runs = {}
    for dual in ("0", "1"):
        monkeypatch.setenv("KDKL_DUAL_DHDW", dual)
        runs[dual] = run_gpu(kdkl, x, w.tau, w.chunk, grad_loss=0.8)
    for key in ("dH", "dW"):
        assert np.array_equal(runs["0"][key], runs["1"][key]), key
    _compare(runs["0"], x, w.tau, grad_loss=0.8)
