"""ctypes binding of libkdkl.so (the C ABI in include/kdkl.h).

Argument marshalling only: every step of the loss runs in the library's CUDA
kernels. PyTorch provides device memory (outputs and the workspace) and the
current stream. There is no CPU fallback: if the library is missing the calls
raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkdkl.so")

KD_OK = 0
STATUS_NAMES = {
    0: "KD_OK", 1: "KD_ERR_INVALID_ARG", 2: "KD_ERR_SHAPE", 3: "KD_ERR_ALIGNMENT",
    4: "KD_ERR_INDEX_RANGE", 5: "KD_ERR_WORKSPACE", 6: "KD_ERR_CUDA", 7: "KD_ERR_TIMEOUT",
    8: "KD_ERR_UNSUPPORTED",
}
KDKL_MAX_K = 512


class KDKLError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s" % (where, STATUS_NAMES.get(code, "status %d" % code)))


class kd_kl_problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int64), ("V", ctypes.c_int64),
                ("K", ctypes.c_int32), ("temperature", ctypes.c_float), ("chunk", ctypes.c_int64)]


class kd_kl_options(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_float), ("scale_tau_sq", ctypes.c_int32),
                ("labels", ctypes.c_void_p)]


class kd_topk_problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int64), ("V", ctypes.c_int64),
                ("K", ctypes.c_int32), ("reserved", ctypes.c_int32)]


KDKL_TOPK_MAX_K = 512


class kd_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


# name -> (restype, argtypes); every symbol include/kdkl.h declares.
_P = ctypes.c_void_p
_SIGS = {
    "kd_kl_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(kd_kl_problem), ctypes.c_int]),
    "kd_kl_forward": (ctypes.c_int, [ctypes.POINTER(kd_kl_problem), _P, _P, _P, _P, _P, _P, _P, _P,
                                     _P, ctypes.c_size_t, _P]),
    "kd_kl_backward": (ctypes.c_int, [ctypes.POINTER(kd_kl_problem), _P, _P, _P, _P, _P, _P,
                                      ctypes.c_float, _P, _P, ctypes.c_int, _P, ctypes.c_size_t,
                                      _P]),
    "kd_kl_forward_ex": (ctypes.c_int, [ctypes.POINTER(kd_kl_problem), ctypes.POINTER(kd_kl_options),
                                        _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                        _P]),
    "kd_kl_backward_ex": (ctypes.c_int, [ctypes.POINTER(kd_kl_problem),
                                         ctypes.POINTER(kd_kl_options), _P, _P, _P, _P, _P, _P, _P,
                                         ctypes.c_float, _P, _P, ctypes.c_int, _P, ctypes.c_size_t,
                                         _P]),
    "kd_kl_backward_reuse": (ctypes.c_int, [ctypes.POINTER(kd_kl_problem),
                                            ctypes.POINTER(kd_kl_options), _P, _P, _P, _P, _P, _P,
                                            ctypes.c_size_t, ctypes.c_float, _P, _P, ctypes.c_int,
                                            _P, ctypes.c_size_t, _P]),
    "kd_kl_forward_noalloc": (ctypes.c_int, [ctypes.POINTER(kd_kl_problem), _P, _P, _P, _P, _P,
                                             _P, _P, _P, _P]),
    "kd_kl_noalloc_check_status": (ctypes.c_int, [_P]),
    "kd_rkl_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(kd_kl_problem)]),
    "kd_rkl_forward": (ctypes.c_int, [ctypes.POINTER(kd_kl_problem), _P, _P, _P, _P, _P, _P, _P,
                                      _P, _P, ctypes.c_size_t, _P]),
    "kd_rkl_backward": (ctypes.c_int, [ctypes.POINTER(kd_kl_problem), _P, _P, _P, _P, _P, _P,
                                       ctypes.c_float, _P, _P, ctypes.c_int, _P, ctypes.c_size_t,
                                       _P]),
    "kd_lmhead_topk_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(kd_topk_problem)]),
    "kd_lmhead_topk": (ctypes.c_int, [ctypes.POINTER(kd_topk_problem), _P, _P, _P, _P, _P,
                                      ctypes.c_size_t, _P]),
    "kd_kl_check_status": (ctypes.c_int, [_P, _P]),
    "kd_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kd_launch_count": (ctypes.c_int64, []),
    "kd_timing_begin": (ctypes.c_int, []),
    "kd_timing_end": (ctypes.c_int, [ctypes.POINTER(kd_kernel_time), ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_int)]),
}

_lib: Optional[ctypes.CDLL] = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError("libkdkl.so not found at %s: build it with "
                               "`python -m lm_head_top_gb300.build`" % path)
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _problem(T, d, V, K, temperature, chunk) -> kd_kl_problem:
    return kd_kl_problem(int(T), int(d), int(V), int(K), float(temperature), int(chunk))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t: torch.Tensor, name: str, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be on a CUDA device" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))


def same_device(dev: torch.device, **tensors) -> None:
    """Every tensor given (None skipped) must live on ``dev``: the library runs
    on the current device with pointers as they are, so a tensor on another
    GPU would be read through the wrong device. Raises before anything runs."""
    for name, t in tensors.items():
        if t is not None and t.device != dev:
            raise ValueError("%s is on %s, expected %s (the device of H)" % (name, t.device, dev))


def _out(t, name, dtype, shape, dev):
    """An output tensor passed in: right dtype, shape, contiguity and device."""
    if t is not None:
        _check(t, name, dtype, shape)
        same_device(dev, **{name: t})
    return t


def kd_status_string(code: int) -> str:
    return load().kd_status_string(int(code)).decode()


def kd_launch_count() -> int:
    return int(load().kd_launch_count())


def kd_kl_workspace_size(T, d, V, K, temperature=1.0, chunk=1024, which=0) -> int:
    p = _problem(T, d, V, K, temperature, chunk)
    return int(load().kd_kl_workspace_size(ctypes.byref(p), int(which)))


def _workspace(p: kd_kl_problem, which: int, device, workspace):
    need = int(load().kd_kl_workspace_size(ctypes.byref(p), which))
    if need == 0:
        raise KDKLError(2, "kd_kl_workspace_size")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    else:
        _check(workspace, "workspace", torch.uint8, (workspace.numel(),))
        same_device(device, workspace=workspace)
    return workspace


def _call(fn_name: str, dev: torch.device, stream, *args):
    """Runs one library call with ``dev`` current (the library works on the
    current device and stream), raising KDKLError on a non-OK status."""
    if stream is not None and stream.device != dev:
        raise ValueError("stream is on %s, expected %s" % (stream.device, dev))
    with torch.cuda.device(dev):
        rc = getattr(load(), fn_name)(*args, _stream_ptr(stream))
    if rc != KD_OK:
        raise KDKLError(rc, fn_name)


def _teacher_args(H, W, topk_idx, topk_logit, mask):
    T, d = H.shape
    V = W.shape[0]
    K = topk_idx.shape[1]
    _check(H, "H", torch.bfloat16, (T, d))
    _check(W, "W", torch.bfloat16, (V, d))
    _check(topk_idx, "topk_idx", torch.int32, (T, K))
    _check(topk_logit, "topk_logit", torch.float32, (T, K))
    if mask is not None:
        _check(mask, "mask", torch.uint8, (T,))
    same_device(H.device, W=W, topk_idx=topk_idx, topk_logit=topk_logit, mask=mask)
    return T, d, V, K, H.device


def kd_kl_forward(H, W, topk_idx, topk_logit, mask=None, *, temperature=1.0, chunk=1024,
                  want_token_kl=False, loss=None, lse=None, token_kl=None, workspace=None,
                  stream=None):
    """Fused forward. Returns (loss [1] fp32, lse [T] fp32, token_kl [T] fp32 or None).
    The work is queued on ``stream`` (default: the current stream of H's device)."""
    T, d, V, K, dev = _teacher_args(H, W, topk_idx, topk_logit, mask)
    p = _problem(T, d, V, K, temperature, chunk)
    workspace = _workspace(p, 0, dev, workspace)
    loss = _out(loss, "loss", torch.float32, (1,), dev)
    lse = _out(lse, "lse", torch.float32, (T,), dev)
    token_kl = _out(token_kl, "token_kl", torch.float32, (T,), dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev) if loss is None else loss
    lse = torch.empty(T, dtype=torch.float32, device=dev) if lse is None else lse
    if want_token_kl and token_kl is None:
        token_kl = torch.empty(T, dtype=torch.float32, device=dev)
    _call("kd_kl_forward", dev, stream, ctypes.byref(p), _ptr(H), _ptr(W), _ptr(topk_idx),
          _ptr(topk_logit), _ptr(mask), _ptr(loss), _ptr(lse), _ptr(token_kl), _ptr(workspace),
          workspace.numel())
    return loss, lse, token_kl


def _grad_outputs(dH, dW, T, V, d, accumulate_dW, dev):
    dH = _out(dH, "dH", torch.bfloat16, (T, d), dev)
    dW = _out(dW, "dW", torch.float32, (V, d), dev)
    dH = torch.empty((T, d), dtype=torch.bfloat16, device=dev) if dH is None else dH
    if dW is None:
        if accumulate_dW:
            raise ValueError("accumulate_dW needs an existing dW")
        dW = torch.empty((V, d), dtype=torch.float32, device=dev)
    return dH, dW


def kd_kl_backward(H, W, topk_idx, topk_logit, mask, lse, *, temperature=1.0, chunk=1024,
                   grad_loss=1.0, dH=None, dW=None, accumulate_dW=False, workspace=None,
                   fwd_workspace=None, stream=None):
    """Fused backward of grad_loss * loss. Returns (dH [T,d] bf16, dW [V,d] fp32).

    ``fwd_workspace``: the workspace the forward on these inputs used. The
    backward then reads the teacher rows that forward prepared instead of
    preparing them again (kd_kl_backward_reuse); topk_idx / topk_logit are
    only shape-checked."""
    T, d, V, K, dev = _teacher_args(H, W, topk_idx, topk_logit, mask)
    _check(lse, "lse", torch.float32, (T,))
    same_device(dev, lse=lse)
    p = _problem(T, d, V, K, temperature, chunk)
    dH, dW = _grad_outputs(dH, dW, T, V, d, accumulate_dW, dev)
    if fwd_workspace is not None:
        _check(fwd_workspace, "fwd_workspace", torch.uint8, (fwd_workspace.numel(),))
        same_device(dev, fwd_workspace=fwd_workspace)
        workspace = _workspace(p, 4, dev, workspace)
        _call("kd_kl_backward_reuse", dev, stream, ctypes.byref(p), None, _ptr(H), _ptr(W),
              _ptr(mask), _ptr(lse), None, _ptr(fwd_workspace), fwd_workspace.numel(),
              float(grad_loss), _ptr(dH), _ptr(dW), 1 if accumulate_dW else 0, _ptr(workspace),
              workspace.numel())
        return dH, dW
    workspace = _workspace(p, 1, dev, workspace)
    _call("kd_kl_backward", dev, stream, ctypes.byref(p), _ptr(H), _ptr(W), _ptr(topk_idx),
          _ptr(topk_logit), _ptr(mask), _ptr(lse), float(grad_loss), _ptr(dH), _ptr(dW),
          1 if accumulate_dW else 0, _ptr(workspace), workspace.numel())
    return dH, dW


def _options(alpha, scale_tau_sq, labels, T, dev):
    if labels is not None:
        _check(labels, "labels", torch.int32, (T,))
        same_device(dev, labels=labels)
    return kd_kl_options(float(alpha), 1 if scale_tau_sq else 0,
                         None if labels is None else labels.data_ptr())


def kd_kl_forward_ex(H, W, topk_idx, topk_logit, mask=None, labels=None, *, temperature=1.0,
                     chunk=1024, alpha=1.0, scale_tau_sq=False, want_token_loss=False,
                     workspace=None, stream=None):
    """Mixed loss alpha*c*KL(tau) + (1-alpha)*CE(labels), c = tau^2 if scale_tau_sq.
    Returns (loss [1], lse [T] at tau, lse1 [T] at temperature 1, token_loss or None)."""
    T, d, V, K, dev = _teacher_args(H, W, topk_idx, topk_logit, mask)
    p = _problem(T, d, V, K, temperature, chunk)
    o = _options(alpha, scale_tau_sq, labels, T, dev)
    workspace = _workspace(p, 2, dev, workspace)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    lse1 = torch.empty(T, dtype=torch.float32, device=dev)
    tok = torch.empty(T, dtype=torch.float32, device=dev) if want_token_loss else None
    _call("kd_kl_forward_ex", dev, stream, ctypes.byref(p), ctypes.byref(o), _ptr(H), _ptr(W),
          _ptr(topk_idx), _ptr(topk_logit), _ptr(mask), _ptr(loss), _ptr(lse), _ptr(lse1),
          _ptr(tok), _ptr(workspace), workspace.numel())
    return loss, lse, lse1, tok


def kd_kl_backward_ex(H, W, topk_idx, topk_logit, mask, labels, lse, lse1, *, temperature=1.0,
                      chunk=1024, alpha=1.0, scale_tau_sq=False, grad_loss=1.0, dH=None, dW=None,
                      accumulate_dW=False, workspace=None, fwd_workspace=None, stream=None):
    """Backward of grad_loss * kd_kl_forward_ex's loss. Returns (dH bf16, dW fp32).
    ``fwd_workspace`` as in kd_kl_backward."""
    T, d, V, K, dev = _teacher_args(H, W, topk_idx, topk_logit, mask)
    _check(lse, "lse", torch.float32, (T,))
    if lse1 is not None:
        _check(lse1, "lse1", torch.float32, (T,))
    same_device(dev, lse=lse, lse1=lse1)
    p = _problem(T, d, V, K, temperature, chunk)
    o = _options(alpha, scale_tau_sq, labels, T, dev)
    dH, dW = _grad_outputs(dH, dW, T, V, d, accumulate_dW, dev)
    if fwd_workspace is not None:
        _check(fwd_workspace, "fwd_workspace", torch.uint8, (fwd_workspace.numel(),))
        same_device(dev, fwd_workspace=fwd_workspace)
        workspace = _workspace(p, 4, dev, workspace)
        _call("kd_kl_backward_reuse", dev, stream, ctypes.byref(p), ctypes.byref(o), _ptr(H),
              _ptr(W), _ptr(mask), _ptr(lse), _ptr(lse1), _ptr(fwd_workspace),
              fwd_workspace.numel(), float(grad_loss), _ptr(dH), _ptr(dW),
              1 if accumulate_dW else 0, _ptr(workspace), workspace.numel())
        return dH, dW
    workspace = _workspace(p, 3, dev, workspace)
    _call("kd_kl_backward_ex", dev, stream, ctypes.byref(p), ctypes.byref(o), _ptr(H), _ptr(W),
          _ptr(topk_idx), _ptr(topk_logit), _ptr(mask), _ptr(lse), _ptr(lse1), float(grad_loss),
          _ptr(dH), _ptr(dW), 1 if accumulate_dW else 0, _ptr(workspace), workspace.numel())
    return dH, dW


def kd_kl_forward_noalloc(H, W, topk_idx, topk_logit, mask=None, *, temperature=1.0,
                          chunk=1024, want_token_kl=False, loss=None, lse=None, token_kl=None,
                          stream=None):
    """Forward for callers that cannot allocate a workspace: the library's own
    fixed scratch array is used instead (see kd_kl_forward_noalloc in kdkl.h).
    Outputs are allocated here only when not passed in."""
    T, d, V, K, dev = _teacher_args(H, W, topk_idx, topk_logit, mask)
    p = _problem(T, d, V, K, temperature, chunk)
    loss = _out(loss, "loss", torch.float32, (1,), dev)
    lse = _out(lse, "lse", torch.float32, (T,), dev)
    token_kl = _out(token_kl, "token_kl", torch.float32, (T,), dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev) if loss is None else loss
    lse = torch.empty(T, dtype=torch.float32, device=dev) if lse is None else lse
    if want_token_kl and token_kl is None:
        token_kl = torch.empty(T, dtype=torch.float32, device=dev)
    _call("kd_kl_forward_noalloc", dev, stream, ctypes.byref(p), _ptr(H), _ptr(W),
          _ptr(topk_idx), _ptr(topk_logit), _ptr(mask), _ptr(loss), _ptr(lse), _ptr(token_kl))
    return loss, lse, token_kl


def kd_kl_noalloc_check_status(device=None, stream=None) -> int:
    """BLOCKING. Device-detected status of the latest kd_kl_forward_noalloc
    call on ``device`` (default: the current device)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    with torch.cuda.device(dev):
        return int(load().kd_kl_noalloc_check_status(_stream_ptr(stream)))


def kd_rkl_workspace_size(T, d, V, K, temperature=1.0) -> int:
    p = _problem(T, d, V, K, temperature, 1)
    return int(load().kd_rkl_workspace_size(ctypes.byref(p)))


def _rkl_args(H, W, topk_idx, topk_logit, mask, temperature, workspace):
    T, d, V, K, dev = _teacher_args(H, W, topk_idx, topk_logit, mask)
    p = _problem(T, d, V, K, temperature, 1)
    if workspace is None:
        need = int(load().kd_rkl_workspace_size(ctypes.byref(p)))
        if need == 0:
            raise KDKLError(2, "kd_rkl_workspace_size")
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    else:
        _check(workspace, "workspace", torch.uint8, (workspace.numel(),))
        same_device(dev, workspace=workspace)
    return p, workspace


def kd_rkl_forward(H, W, topk_idx, topk_logit, mask=None, *, temperature=1.0,
                   want_token_rkl=False, want_grad_z=False, loss=None, token_rkl=None, grad_z=None,
                   workspace=None, stream=None):
    """Reverse KL over the cached ids. Returns (loss [1] fp32, token_rkl [T] fp32 or None,
    grad_z [T,K] fp32 or None)."""
    p, workspace = _rkl_args(H, W, topk_idx, topk_logit, mask, temperature, workspace)
    dev = H.device
    T = H.shape[0]
    loss = _out(loss, "loss", torch.float32, (1,), dev)
    token_rkl = _out(token_rkl, "token_rkl", torch.float32, (T,), dev)
    grad_z = _out(grad_z, "grad_z", torch.float32, tuple(topk_idx.shape), dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev) if loss is None else loss
    if want_token_rkl and token_rkl is None:
        token_rkl = torch.empty(T, dtype=torch.float32, device=dev)
    if want_grad_z and grad_z is None:
        grad_z = torch.empty(tuple(topk_idx.shape), dtype=torch.float32, device=dev)
    _call("kd_rkl_forward", dev, stream, ctypes.byref(p), _ptr(H), _ptr(W), _ptr(topk_idx),
          _ptr(topk_logit), _ptr(mask), _ptr(loss), _ptr(token_rkl), _ptr(grad_z),
          _ptr(workspace), workspace.numel())
    return loss, token_rkl, grad_z


def kd_rkl_backward(H, W, topk_idx, topk_logit, mask=None, *, temperature=1.0, grad_z=None,
                    grad_loss=1.0, dH=None, dW=None, accumulate_dW=False, workspace=None,
                    stream=None):
    """Backward of grad_loss * reverse-KL loss. Returns (dH [T,d] bf16, dW [V,d] fp32).
    grad_z from kd_rkl_forward (same inputs) skips the logit recompute."""
    p, workspace = _rkl_args(H, W, topk_idx, topk_logit, mask, temperature, workspace)
    dev = H.device
    grad_z = _out(grad_z, "grad_z", torch.float32, tuple(topk_idx.shape), dev)
    T, d = H.shape
    dH, dW = _grad_outputs(dH, dW, T, W.shape[0], d, accumulate_dW, dev)
    _call("kd_rkl_backward", dev, stream, ctypes.byref(p), _ptr(H), _ptr(W), _ptr(topk_idx),
          _ptr(topk_logit), _ptr(mask), _ptr(grad_z), float(grad_loss), _ptr(dH), _ptr(dW),
          1 if accumulate_dW else 0, _ptr(workspace), workspace.numel())
    return dH, dW


def kd_lmhead_topk_workspace_size(T, d, V, K) -> int:
    p = kd_topk_problem(int(T), int(d), int(V), int(K), 0)
    return int(load().kd_lmhead_topk_workspace_size(ctypes.byref(p)))


def kd_lmhead_topk(H, W, K, *, topk_idx=None, topk_logit=None, workspace=None, stream=None):
    """Offline teacher cache: the K largest logits of each row of H . W^T and
    their ids, per row by logit descending (ties: smaller id first).
    Returns (topk_idx [T,K] int32, topk_logit [T,K] fp32)."""
    T, d = H.shape
    V = W.shape[0]
    _check(H, "H", torch.bfloat16, (T, d))
    _check(W, "W", torch.bfloat16, (V, d))
    dev = H.device
    same_device(dev, W=W)
    p = kd_topk_problem(int(T), int(d), int(V), int(K), 0)
    need = int(load().kd_lmhead_topk_workspace_size(ctypes.byref(p)))
    if need == 0:
        raise KDKLError(2, "kd_lmhead_topk_workspace_size")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    else:
        _check(workspace, "workspace", torch.uint8, (workspace.numel(),))
        same_device(dev, workspace=workspace)
    topk_idx = _out(topk_idx, "topk_idx", torch.int32, (T, K), dev)
    topk_logit = _out(topk_logit, "topk_logit", torch.float32, (T, K), dev)
    if topk_idx is None:
        topk_idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    if topk_logit is None:
        topk_logit = torch.empty((T, K), dtype=torch.float32, device=dev)
    _call("kd_lmhead_topk", dev, stream, ctypes.byref(p), _ptr(H), _ptr(W), _ptr(topk_idx),
          _ptr(topk_logit), _ptr(workspace), workspace.numel())
    return topk_idx, topk_logit


def kd_kl_check_status(workspace: torch.Tensor, stream=None) -> int:
    """BLOCKING. Device-detected status of the latest call that used ``workspace``."""
    with torch.cuda.device(workspace.device):
        return int(load().kd_kl_check_status(_ptr(workspace), _stream_ptr(stream)))


def kd_timing_begin() -> None:
    load().kd_timing_begin()


def kd_timing_end(max_entries: int = 32):
    """BLOCKING. Returns [(kernel name, launches, total ms)] since kd_timing_begin()."""
    arr = (kd_kernel_time * max_entries)()
    n = ctypes.c_int(0)
    rc = load().kd_timing_end(arr, max_entries, ctypes.byref(n))
    if rc != KD_OK:
        raise KDKLError(rc, "kd_timing_end")
    return [(arr[i].name.decode(), int(arr[i].launches), float(arr[i].total_ms))
            for i in range(min(n.value, max_entries))]
