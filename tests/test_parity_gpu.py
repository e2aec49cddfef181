"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on seeded inputs.

Small and medium shapes are compared element by element over the whole output; they span
several 128-row tiles and ragged tails. The full-size workloads are compared on sampled rows
(every (b, h) with rows 0, 1, 127, 128, N-1 and seeded random rows), in the same launch
configuration the benchmark times, plus properties that hold for every row.
"""
import numpy as np
import pytest

import oracle
from gpu_util import assert_close, attention_aux, run_gpu, to_device
from io_aware_attention_fa2_gb300.inputs import (WORKLOADS, make_qkv, make_workload,
                                                 sample_rows, softmax_scale)

pytestmark = pytest.mark.gpu


def _full_case(B, H, N, d, dtype, causal, seed, scale=None, **kw):
    qb, kb, vb = make_qkv(B, H, N, d, dtype, seed, **kw)
    scale = softmax_scale(d) if scale is None else scale
    o, lse = run_gpu(qb, kb, vb, dtype, causal, scale)
    o_ref, lse_ref = oracle.attention(qb, kb, vb, causal, scale, dtype=dtype)
    a_ref, _ = attention_aux(qb, kb, vb, causal, scale, dtype)
    return assert_close(o, lse, o_ref, lse_ref, "B=%d H=%d N=%d d=%d %s causal=%s" %
                        (B, H, N, d, dtype, causal), dtype, a_ref)


@pytest.mark.parametrize("N", [1, 2, 17, 127, 128, 129, 255, 300, 513])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_shapes_full(N, d, causal, dtype):
    _full_case(2, 3, N, d, dtype, causal, seed=100 + N + d)


@pytest.mark.parametrize("scale", [0.0, -0.09, 1.0, 1e-3])
@pytest.mark.parametrize("causal", [False, True])
def test_scale_values(scale, causal):
    _full_case(1, 2, 200, 64, "bf16", causal, seed=7, scale=scale)


@pytest.mark.parametrize("causal", [False, True])
def test_large_logits_small(causal):
    """Q x8 and 1% of K rows x10 in fp16: scores far beyond exp's fp32 range."""
    _full_case(2, 2, 333, 128, "fp16", causal, seed=8, q_scale=8.0, k_outlier_frac=0.01,
               k_outlier_scale=10.0)


@pytest.mark.parametrize("name", ["tiny_n256_d64", "n1k_d64", "n1k_d64_causal"])
def test_workload_full(name):
    w = WORKLOADS[name]
    qb, kb, vb = make_workload(w)
    o, lse = run_gpu(qb, kb, vb, w.dtype, w.causal, w.scale)
    o_ref, lse_ref = oracle.attention(qb, kb, vb, w.causal, w.scale, dtype=w.dtype)
    assert_close(o, lse, o_ref, lse_ref, name, w.dtype)


@pytest.mark.parametrize("name", ["n8k_d128_causal", "n32k_d128_causal",
                                  "n2000_d128_fp16_stress"])
def test_workload_sampled(name):
    import torch

    from io_aware_attention_fa2_gb300 import binding
    w = WORKLOADS[name]
    qb, kb, vb = make_workload(w)
    q, k, v = (to_device(x, w.dtype) for x in (qb, kb, vb))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=q.device)
    binding.fa_fwd(q, k, v, o, lse, w.causal, w.scale)
    assert binding.device_error() == 0
    per_head = max(4, 4096 // (w.B * w.H))
    rows = sample_rows(w.B, w.H, w.N, per_head, seed=w.seed + 7)
    o_ref, lse_ref = oracle.attention_rows(qb, kb, vb, rows, w.causal, w.scale, dtype=w.dtype)
    rb, rh, ri = (torch.from_numpy(rows[:, c]).cuda() for c in range(3))
    o_rows = o[rb, ri, rh].double().cpu().numpy()
    lse_rows = lse[rb, rh, ri].double().cpu().numpy()
    assert_close(o_rows, lse_rows, o_ref, lse_ref, name, w.dtype)

    # Every row: finite, and each O entry inside the range of the V entries it averages.
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    vf = v.float()
    if w.causal:
        hi = torch.cummax(vf, dim=1).values
        lo = torch.cummin(vf, dim=1).values
    else:
        hi = vf.amax(dim=1, keepdim=True)
        lo = vf.amin(dim=1, keepdim=True)
    of = o.float()
    assert bool((of <= hi + 1e-2).all()) and bool((of >= lo - 1e-2).all())


def test_deterministic_and_stream():
    import torch

    from io_aware_attention_fa2_gb300 import binding
    qb, kb, vb = make_qkv(2, 4, 700, 128, "bf16", seed=9)
    q, k, v = (to_device(x, "bf16") for x in (qb, kb, vb))
    outs = []
    side = torch.cuda.Stream()
    for stream in (None, side):
        o = torch.empty_like(q)
        lse = torch.empty((2, 4, 700), dtype=torch.float32, device=q.device)
        with torch.cuda.stream(stream or torch.cuda.current_stream()):
            binding.fa_fwd(q, k, v, o, lse, True, softmax_scale(128), stream)
        torch.cuda.synchronize()
        outs.append((o.clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_bad_arguments_on_gpu_leave_outputs_untouched():
    import torch

    from io_aware_attention_fa2_gb300 import binding
    q = torch.randn(1, 256, 2, 64, device="cuda").to(torch.bfloat16)
    k, v = torch.randn_like(q), torch.randn_like(q)
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 2, 256, device="cuda")
    lib = binding.load_library()
    st = torch.cuda.current_stream().cuda_stream
    # output aliasing an input
    assert lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), q.data_ptr(), lse.data_ptr(),
                      1, 2, 256, 64, 0, 0.125, 0, st) == -5
    # unsupported head dimension
    assert lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      1, 4, 256, 32, 0, 0.125, 0, st) == -2
    torch.cuda.synchronize()
    assert int(o.abs().sum()) == 0 and float(lse.abs().sum()) == 0.0
    with pytest.raises(binding.FaError):
        binding.fa_fwd(q, k, v, q, lse, False, 0.125)


def test_user_api_host_and_device_tensors():
    import torch

    from io_aware_attention_fa2_gb300 import attention_forward
    qb, kb, vb = make_qkv(1, 2, 300, 64, "fp16", seed=10)
    host = [torch.from_numpy(x.view(np.int16)).view(torch.float16).pin_memory()
            for x in (qb, kb, vb)]
    o_h, lse_h = attention_forward(*host, causal=True)
    o_d, lse_d = attention_forward(*(t.cuda() for t in host), causal=True)
    assert not o_h.is_cuda and torch.equal(o_h, o_d.cpu()) and torch.equal(lse_h, lse_d.cpu())
    o_ref, lse_ref = oracle.attention(qb, kb, vb, True, softmax_scale(64), dtype="fp16")
    assert_close(o_h.double().numpy(), lse_h.double().numpy(), o_ref, lse_ref, "user API",
                 "fp16")


@pytest.mark.parametrize("B,H,N,d,causal,pinned", [
    (1, 4, 200, 64, True, True), (3, 4, 1000, 128, False, True), (5, 4, 333, 128, True, False),
    (2, 16, 8192, 128, True, True),     # 8 head groups of 2 heads
    (3, 11, 8192, 64, False, True),     # 8 unequal groups (11 has no divisor from 4 to 8)
    (1, 12, 16384, 128, True, False)])  # 6 groups of 2 heads, pageable host memory
def test_host_entry_matches_device_path(B, H, N, d, causal, pinned):
    """fa_fwd_host (host buffers, head groups packed by pitched copies, copies overlapping the
    kernels) gives exactly the device path's O and LSE: the same kernel on the same values."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed=8100 + B + N)
    hq, hk, hv = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) for x in (qb, kb, vb))
    if pinned:
        hq, hk, hv = (t.pin_memory() for t in (hq, hk, hv))
    o_h, l_h = binding.attention_forward(hq, hk, hv, causal=causal)
    q, k, v = (t.cuda() for t in (hq, hk, hv))
    o_d, l_d = binding.attention_forward(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    assert torch.equal(o_h.view(torch.int16), o_d.cpu().view(torch.int16))
    assert torch.equal(l_h, l_d.cpu())


def test_many_small_heads_full():
    """B x H = 2048 heads of 128 rows (2048 units of one Q tile each, many dispatch groups),
    every output row against the oracle."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    B, H, N, d = 64, 32, 128, 64
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed=8300)
    q, k, v = (to_device(x, "bf16") for x in (qb, kb, vb))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    binding.fa_fwd(q, k, v, o, lse, True, softmax_scale(d))
    assert binding.device_error() == 0
    o_ref, lse_ref = oracle.attention(qb, kb, vb, True, softmax_scale(d), dtype="bf16")
    assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref,
                 "64x32 heads of 128", "bf16")


def test_long_sequence_d64_sampled():
    """N = 32768 with d = 64 (256 K/V tiles for the last Q block), causal; sampled rows."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    B, H, N, d = 1, 2, 32768, 64
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed=8400)
    q, k, v = (to_device(x, "bf16") for x in (qb, kb, vb))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    binding.fa_fwd(q, k, v, o, lse, True, softmax_scale(d))
    assert binding.device_error() == 0
    rows = sample_rows(B, H, N, 48, seed=8401)
    o_ref, lse_ref = oracle.attention_rows(qb, kb, vb, rows, True, softmax_scale(d), dtype="bf16")
    rb, rh, ri = (torch.from_numpy(rows[:, c]).cuda() for c in range(3))
    assert_close(o[rb, ri, rh].double().cpu().numpy(), lse[rb, rh, ri].double().cpu().numpy(),
                 o_ref, lse_ref, "N=32768 d=64", "bf16")


@pytest.mark.parametrize("window,lens,causal", [((100, 0), None, True),
                                                ((-1, -1), [1000, 333], False),
                                                ((64, 64), None, False),
                                                ((300, -1), [1000, 900], True)])
def test_masked_host_entry_matches_device_path(window, lens, causal):
    """fa_fwd_host_masked (host buffers with the window and key-length masks) gives exactly the
    device path's O and LSE."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    B, H, N, d = 2, 6, 1000, 128
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed=8700 + (lens[1] if lens else 0))
    hq, hk, hv = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
                  for x in (qb, kb, vb))
    lens_t = None if lens is None else torch.tensor(lens, dtype=torch.int32)
    o_h, l_h = binding.attention_forward(hq, hk, hv, causal=causal, window=window,
                                         seqlens_k=lens_t)
    o_d, l_d = binding.attention_forward(hq.cuda(), hk.cuda(), hv.cuda(), causal=causal,
                                         window=window,
                                         seqlens_k=None if lens_t is None else lens_t.cuda())
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    assert torch.equal(o_h.view(torch.int16), o_d.cpu().view(torch.int16))
    assert torch.equal(l_h, l_d.cpu())
    o_ref, lse_ref = oracle.attention(qb, kb, vb, causal, softmax_scale(d), dtype="bf16",
                                      window=window, seqlens_k=lens)
    assert_close(o_h.double().numpy(), l_h.double().numpy(), o_ref, lse_ref, "host masked",
                 "bf16")


def test_non_device_pointers_are_refused_before_launch():
    """Host memory passed where device memory is expected returns FA_ERR_POINTER and launches
    nothing; device memory of the current device passes. The case checked puts the LSE output
    in pinned host memory, which a kernel could even write safely (mapped host memory), so the
    test runs nothing that could fault should the check ever let it through."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    lib = binding.load_library()
    B, H, N, d = 1, 2, 256, 64
    q = torch.randn(B, N, H, d, device="cuda").to(torch.bfloat16)
    k, v, o = torch.randn_like(q), torch.randn_like(q), torch.zeros_like(q)
    lse = torch.zeros(B, H, N, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    bad_lse = torch.zeros(B, H, N).pin_memory()
    assert lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), bad_lse.data_ptr(),
                      B, H, N, d, 0, 0.125, 0, st) == -12
    torch.cuda.synchronize()
    assert int(o.view(torch.int16).abs().sum()) == 0          # nothing ran
    assert float(bad_lse.abs().sum()) == 0.0
    assert lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B,
                      H, N, d, 0, 0.125, 0, st) == 0
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    assert lib.fa_error_string(-12) == (
        b"a device-side argument is not device memory of the current device")
