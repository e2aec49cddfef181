"""fa_fwd_splitkv_noalloc: the split-K/V forward for callers that cannot allocate device memory
when they call (a plugin inside a host that owns the device-memory budget, or a latency-
critical loop that cannot afford an allocation). It uses the library's built-in 8 MiB buffer
instead of a caller workspace.

Checked through the C ABI against fa_fwd_splitkv with a workspace PyTorch allocates, on two
calls in a row: the second call has a different shape and reuses the buffer the first one left
behind. Both run the same kernels on the same values, so the outputs must be bit-identical.
A further check makes several calls and reads the device's free memory before and after: a
call that allocated would lower it. This file is collected last so that a run stopping at the
first failure has run every other test before it; it also passes alone in a fresh process.
"""
import ctypes

import pytest

from gpu_util import to_device
from io_aware_attention_fa2_gb300.inputs import make_qkv, softmax_scale

pytestmark = pytest.mark.gpu

FA_ERR_WORKSPACE = -11
BUFFER_BYTES = 8 << 20


def _lib():
    from io_aware_attention_fa2_gb300 import binding
    lib = binding.load_library()
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn = lib.fa_fwd_splitkv_noalloc
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, f32, i32, i32,
                   vp]
    fn.restype = i32
    return lib


def _call_noalloc(lib, q, k, v, o, lse, causal, splits):
    import torch
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    dtype = 0 if q.dtype == torch.bfloat16 else 1
    return lib.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, H, Nq, Nk, d, int(causal), -1, -1,
                                      None, softmax_scale(d), dtype, splits,
                                      torch.cuda.current_stream().cuda_stream)


def test_two_calls_match_splitkv_with_own_workspace():
    import torch

    from io_aware_attention_fa2_gb300 import binding
    lib = _lib()
    cases = [  # (B, H, Nq, Nk, d, dtype, causal, splits, seed)
        (2, 4, 3, 5000, 128, "bf16", True, 6, 901),
        (1, 3, 1, 1800, 64, "fp16", False, 4, 902),
    ]
    for B, H, Nq, Nk, d, dtype, causal, splits, seed in cases:
        assert binding.splitkv_workspace_size(B, H, Nq, d, splits) <= BUFFER_BYTES
        qb, kb, vb = make_qkv(B, H, Nq, d, dtype, seed, Nk=Nk)
        q, k, v = (to_device(x, dtype) for x in (qb, kb, vb))
        o_ref, o = torch.empty_like(q), torch.full_like(q, float("nan"))
        lse_ref = torch.empty(B, H, Nq, device="cuda")
        lse = torch.full_like(lse_ref, float("nan"))
        binding.fa_fwd_splitkv(q, k, v, o_ref, lse_ref, causal, softmax_scale(d), splits)
        assert _call_noalloc(lib, q, k, v, o, lse, causal, splits) == 0
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse, lse_ref)


def test_calls_allocate_no_device_memory():
    import torch

    from io_aware_attention_fa2_gb300 import binding
    lib = _lib()
    B, H, Nq, Nk, d, splits = 1, 8, 2, 8192, 128, 8
    qb, kb, vb = make_qkv(B, H, Nq, d, "bf16", 903, Nk=Nk)
    q, k, v = (to_device(x, "bf16") for x in (qb, kb, vb))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Nq, device="cuda")
    assert _call_noalloc(lib, q, k, v, o, lse, True, splits) == 0      # set-up done here
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(8):
        assert _call_noalloc(lib, q, k, v, o, lse, True, splits) == 0
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert binding.device_error() == 0
    assert free_after >= free_before, (free_before, free_after)


def test_parts_beyond_the_buffer_are_rejected():
    import torch
    lib = _lib()
    # 64 heads x 256 queries x 128 parts x (128 + 1) x 4 bytes is far more than 8 MiB; the
    # size check returns before anything is enqueued, so small tensors are enough here.
    q = torch.zeros(1, 256, 64, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 64, 256, device="cuda")
    assert _call_noalloc(lib, q, q, q, o, lse, False, 128) == FA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert float(o.float().abs().sum()) == 0.0 and float(lse.abs().sum()) == 0.0
