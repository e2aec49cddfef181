"""Fused exact attention forward for GB300 (sm_103a).

O = softmax(scale * Q K^T [+ causal mask]) V over [B, N, H, d] bf16/fp16 tensors, computed
tile by tile with online softmax so that the N x N score matrix never reaches HBM, plus the
per-row fp32 log-sum-exp. The computation runs in hand-written CUDA kernels behind a C ABI
(``include/fa.h``); this package is a thin ctypes binding over that library.

Importing the package does not load the CUDA library; the first call does, and raises if the
library has not been built (there is no fallback path).
"""
from .binding import (FaError, attention_backward, attention_forward, available,
                      bwd_workspace_size, device_error, error_string, fa_bwd, fa_fwd,
                      fa_fwd_splitkv, library_path, load_library, splitkv_num_splits,
                      splitkv_workspace_size)

__all__ = ["FaError", "attention_backward", "attention_forward", "available",
           "bwd_workspace_size", "device_error", "error_string", "fa_bwd", "fa_fwd",
           "fa_fwd_splitkv", "library_path", "load_library", "splitkv_num_splits",
           "splitkv_workspace_size"]
