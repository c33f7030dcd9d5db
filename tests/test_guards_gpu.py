"""Out-of-bounds writes, unwritten outputs and reads of uninitialised
workspace, checked without a sanitizer. Every output and the workspace sit
between guard bytes that must survive each call, and both start filled with
0xFF bytes (a NaN pattern). The results must then equal, bit for bit, those
of a clean run with fresh buffers; every path here is bitwise deterministic.
Shapes are ragged in every dimension and cover both backward plans
(vocabulary slabs and token chunks)."""
import pytest
import torch

from lm_head_top_gb300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

GUARD = 1024   # bytes on each side; keeps the 16-byte alignment of the slice
CANARY = 0xA5
POISON = 0xFF


@pytest.fixture(scope="module")
def kdkl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_top_gb300 import kdkl as m
    m.load()
    return m


class Guarded:
    """A device buffer of `nbytes` between two guard regions."""

    def __init__(self, nbytes: int):
        self.n = int(nbytes)
        self.buf = torch.full((GUARD + self.n + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.buf[GUARD:GUARD + self.n].fill_(POISON)

    def as_(self, dtype, shape):
        return self.buf[GUARD:GUARD + self.n].view(dtype).view(shape)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        return bool((self.buf[:GUARD] == CANARY).all()) and bool(
            (self.buf[GUARD + self.n:] == CANARY).all())


def _bytes(dtype, shape):
    n = 1
    for s in shape:
        n *= s
    return n * torch.tensor([], dtype=dtype).element_size()


def _guarded(dtype, shape):
    g = Guarded(_bytes(dtype, shape))
    return g, g.as_(dtype, shape)


def _inputs(T, d, V, K, seed):
    w = WORKLOADS["small"].with_(T=T, d=d, V=V, K=K, seq_len=max(T // 3, 1), pad_frac=0.25)
    x = make_inputs(w, seed=seed)
    return {k: v.cuda() for k, v in x.items()}


def _same(a, b):
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8)) if a.dtype == torch.bfloat16 \
        else torch.equal(a, b)


@pytest.mark.parametrize("shape", [
    (131, 72, 1000, 7, 50, 2.0),     # vocabulary slabs, ragged everywhere
    (700, 64, 300, 5, 200, 1.0),     # token chunks (T > V)
    (257, 136, 2100, 33, 300, 0.7),  # several slabs, K > 32
])
def test_kl_paths_stay_in_bounds(kdkl, shape):
    T, d, V, K, chunk, tau = shape
    g = _inputs(T, d, V, K, seed=31)
    args = (g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"])
    guards = []
    gl, loss = _guarded(torch.float32, (1,))
    gs, lse = _guarded(torch.float32, (T,))
    gk, tkl = _guarded(torch.float32, (T,))
    gwf, wsf = _guarded(torch.uint8, (kdkl.kd_kl_workspace_size(T, d, V, K, tau, chunk, 0),))
    gh, dH = _guarded(torch.bfloat16, (T, d))
    gw, dW = _guarded(torch.float32, (V, d))
    gwb, wsb = _guarded(torch.uint8, (kdkl.kd_kl_workspace_size(T, d, V, K, tau, chunk, 1),))
    guards += [gl, gs, gk, gwf, gh, gw, gwb]
    kdkl.kd_kl_forward(*args, temperature=tau, chunk=chunk, want_token_kl=True, loss=loss, lse=lse,
                       token_kl=tkl, workspace=wsf)
    kdkl.kd_kl_backward(*args, lse, temperature=tau, chunk=chunk, grad_loss=0.9, dH=dH, dW=dW,
                        workspace=wsb)
    assert all(x.intact() for x in guards)
    assert kdkl.kd_kl_check_status(wsf) == 0 and kdkl.kd_kl_check_status(wsb) == 0
    c_loss, c_lse, c_tkl = kdkl.kd_kl_forward(*args, temperature=tau, chunk=chunk,
                                              want_token_kl=True)
    c_dH, c_dW = kdkl.kd_kl_backward(*args, c_lse, temperature=tau, chunk=chunk, grad_loss=0.9)
    torch.cuda.synchronize()
    for a, b in ((loss, c_loss), (lse, c_lse), (tkl, c_tkl), (dH, c_dH), (dW, c_dW)):
        assert _same(a, b)
    assert torch.isfinite(dW).all() and torch.isfinite(dH.float()).all()


def test_mixed_loss_stays_in_bounds(kdkl):
    T, d, V, K, chunk, tau = 131, 72, 1000, 7, 50, 2.0
    g = _inputs(T, d, V, K, seed=32)
    labels = torch.randint(0, V, (T,), dtype=torch.int32, device="cuda")
    args = (g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"], labels)
    kw = dict(temperature=tau, chunk=chunk, alpha=0.4, scale_tau_sq=True)
    gwf, wsf = _guarded(torch.uint8, (kdkl.kd_kl_workspace_size(T, d, V, K, tau, chunk, 2),))
    gh, dH = _guarded(torch.bfloat16, (T, d))
    gw, dW = _guarded(torch.float32, (V, d))
    gwb, wsb = _guarded(torch.uint8, (kdkl.kd_kl_workspace_size(T, d, V, K, tau, chunk, 3),))
    loss, lse, lse1, tok = kdkl.kd_kl_forward_ex(*args, want_token_loss=True, workspace=wsf, **kw)
    kdkl.kd_kl_backward_ex(*args, lse, lse1, dH=dH, dW=dW, workspace=wsb, **kw)
    assert all(x.intact() for x in (gwf, gh, gw, gwb))
    c_loss, c_lse, c_lse1, c_tok = kdkl.kd_kl_forward_ex(*args, want_token_loss=True, **kw)
    c_dH, c_dW = kdkl.kd_kl_backward_ex(*args, c_lse, c_lse1, **kw)
    torch.cuda.synchronize()
    for a, b in ((loss, c_loss), (lse, c_lse), (lse1, c_lse1), (tok, c_tok), (dH, c_dH),
                 (dW, c_dW)):
        assert _same(a, b)


@pytest.mark.parametrize("shape", [(131, 72, 1000, 7), (300, 1160, 3000, 40)])
def test_reverse_kl_stays_in_bounds(kdkl, shape):
    T, d, V, K = shape
    tau = 1.3
    g = _inputs(T, d, V, K, seed=33)
    args = (g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"])
    gl, loss = _guarded(torch.float32, (1,))
    gt, trkl = _guarded(torch.float32, (T,))
    gz, gradz = _guarded(torch.float32, (T, K))
    gws, ws = _guarded(torch.uint8, (kdkl.kd_rkl_workspace_size(T, d, V, K, tau),))
    gh, dH = _guarded(torch.bfloat16, (T, d))
    gw, dW = _guarded(torch.float32, (V, d))
    kdkl.kd_rkl_forward(*args, temperature=tau, loss=loss, token_rkl=trkl, grad_z=gradz,
                        workspace=ws)
    kdkl.kd_rkl_backward(*args, temperature=tau, grad_z=gradz, dH=dH, dW=dW, workspace=ws)
    assert all(x.intact() for x in (gl, gt, gz, gws, gh, gw))
    assert kdkl.kd_kl_check_status(ws) == 0
    c_loss, c_trkl, c_gz = kdkl.kd_rkl_forward(*args, temperature=tau, want_token_rkl=True,
                                               want_grad_z=True)
    c_dH, c_dW = kdkl.kd_rkl_backward(*args, temperature=tau, grad_z=c_gz)
    torch.cuda.synchronize()
    for a, b in ((loss, c_loss), (trkl, c_trkl), (gradz, c_gz), (dH, c_dH), (dW, c_dW)):
        assert _same(a, b)


@pytest.mark.parametrize("shape", [(300, 200, 5000, 50), (517, 72, 3001, 256)])
def test_topk_producer_stays_in_bounds(kdkl, shape):
    T, d, V, K = shape
    g = _inputs(T, d, V, 4, seed=34)
    gi, idx = _guarded(torch.int32, (T, K))
    gv, val = _guarded(torch.float32, (T, K))
    gws, ws = _guarded(torch.uint8, (kdkl.kd_lmhead_topk_workspace_size(T, d, V, K),))
    kdkl.kd_lmhead_topk(g["H"], g["W"], K, topk_idx=idx, topk_logit=val, workspace=ws)
    assert all(x.intact() for x in (gi, gv, gws))
    assert kdkl.kd_kl_check_status(ws) == 0
    c_idx, c_val = kdkl.kd_lmhead_topk(g["H"], g["W"], K)
    torch.cuda.synchronize()
    assert torch.equal(idx, c_idx) and torch.equal(val, c_val)
