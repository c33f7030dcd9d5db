"""Fused chunked KL distillation loss (LM head x offline teacher top-K) for GB300.

The compute path is the CUDA library ``libkdkl.so`` (C ABI in
``include/kdkl.h``); ``kdkl`` is its ctypes binding and ``inputs`` the seeded
synthetic input generator.
"""
from .kdkl import (KDKLError, kd_kl_backward, kd_kl_check_status, kd_kl_forward,  # noqa: F401
                   kd_kl_workspace_size, kd_launch_count, kd_lmhead_topk,
                   kd_lmhead_topk_workspace_size, kd_rkl_backward, kd_rkl_forward,
                   kd_rkl_workspace_size, kd_status_string, kd_timing_begin, kd_timing_end)
