"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, rejects bad arguments before touching the device, and sizes a
workspace that grows linearly in T with no T x V term."""
import ctypes
import os
import re

import pytest

from lm_head_top_gb300 import kdkl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def _declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"\b(kd_[a-z0-9_]+)\s*\(", src):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(kdkl.LIB_PATH):
        from lm_head_top_gb300 import build
        build.build()
    return kdkl.load()


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"kd_kl_forward", "kd_kl_backward", "kd_kl_workspace_size", "kd_kl_check_status",
            "kd_status_string"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(kdkl._SIGS) == names


def test_status_strings(lib):
    for code, name in kdkl.STATUS_NAMES.items():
        assert kdkl.kd_status_string(code) == name


def test_problem_struct_layout():
    assert ctypes.sizeof(kdkl.kd_kl_problem) == 40
    assert kdkl.kd_kl_problem.K.offset == 24 and kdkl.kd_kl_problem.chunk.offset == 32


def _fwd(lib, p, H=16, W=16, idx=16, logit=16, ws=256, ws_bytes=1 << 30):
    P = ctypes.c_void_p
    return lib.kd_kl_forward(ctypes.byref(p), P(H), P(W), P(idx), P(logit), None, P(64), P(128),
                             None, P(ws), ws_bytes, None)


def _bwd(lib, p, **kw):
    P = ctypes.c_void_p
    return lib.kd_kl_backward(ctypes.byref(p), P(16), P(16), P(16), P(16), None, P(64), 1.0,
                              P(kw.get("dH", 4096)), P(kw.get("dW", 8192)), 0, P(256), 1 << 30,
                              None)


@pytest.mark.parametrize("field,value,code", [
    ("d", 12, 3),            # d % 8 != 0 -> KD_ERR_ALIGNMENT
    ("d", 0, 2),             # d < 8 -> KD_ERR_SHAPE
    ("K", 0, 2),
    ("K", 513, 2),           # > KDKL_MAX_K
    ("K", 101, 2),           # K > V
    ("T", -1, 2),
    ("temperature", 0.0, 1),
    ("temperature", float("inf"), 1),
    ("chunk", 0, 1),
])
def test_argument_errors_are_synchronous(lib, field, value, code):
    p = kdkl.kd_kl_problem(10, 16, 100, 4, 1.0, 8)
    setattr(p, field, value)
    assert _fwd(lib, p) == code
    assert _bwd(lib, p) == code
    assert lib.kd_kl_workspace_size(ctypes.byref(p), 0) == 0


def test_pointer_errors(lib):
    p = kdkl.kd_kl_problem(10, 16, 100, 4, 1.0, 8)
    assert _fwd(lib, p, ws=0) == 5            # KD_ERR_WORKSPACE
    assert _fwd(lib, p, H=0) == 1             # KD_ERR_INVALID_ARG
    assert _fwd(lib, p, H=8) == 3             # H not 16-byte aligned
    assert _fwd(lib, p, idx=2) == 3
    assert _bwd(lib, p, dW=0) == 1
    assert _bwd(lib, p, dH=24) == 3


def test_valid_call_without_device_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    p = kdkl.kd_kl_problem(10, 16, 100, 4, 1.0, 8)
    assert _fwd(lib, p) in (6, 8)  # KD_ERR_CUDA or KD_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["llama3b_8k", "gptoss20b_32k", "toyproj_256k"])
def test_workspace_linear_in_T_no_TxV(lib, name):
    from lm_head_top_gb300.inputs import WORKLOADS
    w = WORKLOADS[name]
    for which in (0, 1):
        sizes = [kdkl.kd_kl_workspace_size(T, w.d, w.V, w.K, 1.0, w.chunk, which)
                 for T in (w.T // 4, w.T // 2, w.T)]
        assert all(s > 0 for s in sizes)
        # a T x V term in bf16 would be at least 2*T*V bytes
        assert sizes[-1] < 0.5 * 2 * w.T * w.V, (which, sizes)
    # the gradient-of-logits buffer stays within chunk x V bf16 (+ tile padding)
    bwd = kdkl.kd_kl_workspace_size(w.T, w.d, w.V, w.K, 1.0, w.chunk, 1)
    # sorted teacher (id, p), the fp32 dH accumulator, and the compaction of
    # the counted tokens (row maps and H's counted rows in bf16)
    per_token = 2 * 4 * w.K + 4 * w.d + 2 * 4 + 2 * w.d
    g_budget = 2 * w.chunk * w.V * 1.07 + 2 * 256 * w.T + 2 * 128 * w.V
    assert bwd <= w.T * per_token + g_budget + (1 << 20)


def _rkl_fwd(lib, p, H=16, ws=256, loss=64):
    P = ctypes.c_void_p
    return lib.kd_rkl_forward(ctypes.byref(p), P(H), P(16), P(16), P(16), None, P(loss), None,
                              None, P(ws), 1 << 30, None)


def _rkl_bwd(lib, p, dH=4096, dW=8192, g=1.0):
    P = ctypes.c_void_p
    return lib.kd_rkl_backward(ctypes.byref(p), P(16), P(16), P(16), P(16), None, None, g, P(dH),
                               P(dW), 0, P(256), 1 << 30, None)


@pytest.mark.parametrize("field,value,code", [
    ("d", 12, 3), ("d", 0, 2), ("K", 0, 2), ("K", 513, 2), ("K", 101, 2), ("T", -1, 2),
    ("temperature", 0.0, 1), ("temperature", float("nan"), 1),
])
def test_rkl_argument_errors_are_synchronous(lib, field, value, code):
    p = kdkl.kd_kl_problem(10, 16, 100, 4, 1.0, 1)
    setattr(p, field, value)
    assert _rkl_fwd(lib, p) == code
    assert _rkl_bwd(lib, p) == code
    assert lib.kd_rkl_workspace_size(ctypes.byref(p)) == 0


def test_rkl_pointer_errors_and_workspace(lib):
    p = kdkl.kd_kl_problem(10, 16, 100, 4, 1.0, 1)
    assert _rkl_fwd(lib, p, ws=0) == 5
    assert _rkl_fwd(lib, p, H=0) == 1
    assert _rkl_fwd(lib, p, loss=0) == 1
    assert _rkl_fwd(lib, p, H=8) == 3
    assert _rkl_bwd(lib, p, dW=0) == 1
    assert _rkl_bwd(lib, p, dH=24) == 3
    assert _rkl_bwd(lib, p, g=float("inf")) == 1
    # linear in T (no T x V term): per pair the gradient, z, two sort buffers and
    # the dW partials (2 rows of d fp32 per 256 pairs); 8 bytes per vocabulary row
    T, d, V, K = 32768, 2880, 201088, 100
    sizes = [kdkl.kd_rkl_workspace_size(t, d, V, K) for t in (T // 4, T // 2, T)]
    assert sizes[0] < sizes[1] < sizes[2]
    per_pair = 4 * 6 + 2 * d * 4 / 256 + 1  # + radix histograms (<= 1 byte per pair)
    assert sizes[2] <= T * K * per_pair + 8 * (V + 1) + T + (1 << 20)
    assert abs((sizes[2] - sizes[1]) - (sizes[1] - sizes[0]) * 2) < (1 << 20)
    # T * K must stay below 2^31
    assert kdkl.kd_rkl_workspace_size(1 << 24, 64, 1000, 200) == 0


# ---- mixed loss (kd_kl_forward_ex / kd_kl_backward_ex): option checks come
# back synchronously, before any device call.

def _opts(alpha=0.5, sq=0, labels=64):
    return kdkl.kd_kl_options(alpha, sq, labels)


def _fwd_ex(lib, p, o, lse1=192):
    P = ctypes.c_void_p
    return lib.kd_kl_forward_ex(ctypes.byref(p), None if o is None else ctypes.byref(o), P(16),
                                P(16), P(16), P(16), None, P(64), P(128), P(lse1), None, P(256),
                                1 << 30, None)


def _bwd_ex(lib, p, o, lse1=192):
    P = ctypes.c_void_p
    return lib.kd_kl_backward_ex(ctypes.byref(p), None if o is None else ctypes.byref(o), P(16),
                                 P(16), P(16), P(16), None, P(64), P(lse1), 1.0, P(4096),
                                 P(8192), 0, P(256), 1 << 30, None)


def test_mixed_loss_option_errors_are_synchronous(lib):
    p = kdkl.kd_kl_problem(10, 16, 100, 4, 2.0, 8)
    for fn in (_fwd_ex, _bwd_ex):
        assert fn(lib, p, None) == 1                          # no options
        assert fn(lib, p, _opts(alpha=1.5)) == 1              # alpha outside [0, 1]
        assert fn(lib, p, _opts(alpha=float("nan"))) == 1
        assert fn(lib, p, _opts(alpha=0.5, labels=0)) == 1    # CE term without labels
        assert fn(lib, p, _opts(alpha=0.5, labels=2)) == 3    # labels not 4-byte aligned
        assert fn(lib, p, _opts(), lse1=0) == 1               # tau != 1 needs lse1
    bad = kdkl.kd_kl_problem(10, 12, 100, 4, 2.0, 8)          # d % 8 != 0, before the options
    assert _fwd_ex(lib, bad, _opts(alpha=1.5)) == 3
    # alpha == 1 needs neither labels nor lse1; the call then reaches the device
    import torch
    if not torch.cuda.is_available():
        assert _fwd_ex(lib, p, _opts(alpha=1.0, labels=0)) in (6, 8)
    assert lib.kd_kl_workspace_size(ctypes.byref(p), 2) > 0
    assert lib.kd_kl_workspace_size(ctypes.byref(p), 3) > 0


# ---- offline top-K producer (kd_lmhead_topk)

def _topk(lib, p, H=16, W=16, idx=64, val=128, ws=256, ws_bytes=1 << 30):
    P = ctypes.c_void_p
    return lib.kd_lmhead_topk(ctypes.byref(p), P(H), P(W), P(idx), P(val), P(ws), ws_bytes, None)


@pytest.mark.parametrize("field,value,code", [
    ("K", 0, 2), ("K", 513, 2),          # 1..KDKL_TOPK_MAX_K
    ("K", 101, 2),                       # K > V
    ("d", 12, 3), ("d", 4, 2), ("T", -1, 2), ("V", 0, 2),
])
def test_topk_argument_errors_are_synchronous(lib, field, value, code):
    # V = 1000 unless the case is K > V
    p = kdkl.kd_topk_problem(10, 16, 100 if (field, value) == ("K", 101) else 1000, 4, 0)
    setattr(p, field, value)
    assert _topk(lib, p) == code
    assert lib.kd_lmhead_topk_workspace_size(ctypes.byref(p)) == 0


def test_topk_pointer_errors(lib):
    p = kdkl.kd_topk_problem(10, 16, 100, 4, 0)
    assert _topk(lib, p, ws=0) == 5
    assert _topk(lib, p, H=0) == 1
    assert _topk(lib, p, W=0) == 1
    assert _topk(lib, p, idx=0) == 1
    assert _topk(lib, p, H=8) == 3
    assert _topk(lib, p, idx=2) == 3
    import torch
    if not torch.cuda.is_available():
        assert _topk(lib, p) in (6, 8)   # a valid call reaches the (absent) device
    # the workspace grows linearly in T
    s = [kdkl.kd_lmhead_topk_workspace_size(t, 2880, 201088, 100) for t in (8192, 16384, 32768)]
    assert s[0] < s[1] < s[2] and abs((s[2] - s[1]) - 2 * (s[1] - s[0])) < (1 << 20)


def test_backward_reuse_needs_a_known_forward_workspace(lib):
    """kd_kl_backward_reuse reads the teacher rows a forward call prepared; a
    workspace no forward filled for this problem is refused on the host,
    before anything is queued (no device call happens here)."""
    P = ctypes.c_void_p
    p = kdkl.kd_kl_problem(10, 16, 100, 4, 1.0, 8)
    need = lib.kd_kl_workspace_size(ctypes.byref(p), 4)
    assert 0 < need < lib.kd_kl_workspace_size(ctypes.byref(p), 1)

    def call(fwd_ws):
        return lib.kd_kl_backward_reuse(ctypes.byref(p), None, P(16), P(16), None, P(64), None,
                                        fwd_ws, 1 << 20, 1.0, P(4096), P(8192), 0, P(256),
                                        need, None)
    assert call(None) == 1            # KD_ERR_INVALID_ARG: no forward workspace
    assert call(P(1 << 20)) == 1      # never filled by a forward call
    # ordinary argument checks still come first
    bad = kdkl.kd_kl_problem(10, 12, 100, 4, 1.0, 8)
    assert lib.kd_kl_backward_reuse(ctypes.byref(bad), None, P(16), P(16), None, P(64), None,
                                    P(1 << 20), 1 << 20, 1.0, P(4096), P(8192), 0, P(256), need,
                                    None) == 3


def test_binding_refuses_tensors_on_another_device():
    """The binding runs each call with H's device current; a tensor elsewhere
    is refused before anything is launched."""
    import torch
    a = torch.zeros(4, dtype=torch.uint8)
    kdkl.same_device(a.device, x=a, y=None)
    with pytest.raises(ValueError, match="expected"):
        kdkl.same_device(a.device, x=torch.zeros(4, dtype=torch.uint8, device="meta"))
