"""Parity of the padding and sliding-window masks (fa_fwd_masked) with the fp64 oracle.

Rows with no visible key must come out as O = 0 and LSE = -inf on both sides; every other row
is held to the same tolerances as the unmasked path.
"""
import numpy as np
import pytest

import oracle
from gpu_util import MAX_ABS_LSE, REL_L2_O, o_bound, to_device
from io_aware_attention_fa2_gb300.inputs import (WORKLOADS, make_qkv, make_workload,
                                                 sample_rows, softmax_scale)

pytestmark = pytest.mark.gpu


def run_masked(qb, kb, vb, dtype, causal, window, lens):
    import torch

    from io_aware_attention_fa2_gb300 import binding
    q, k, v = (to_device(x, dtype) for x in (qb, kb, vb))
    B, N, H, d = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    lens_t = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=q.device)
    binding.fa_fwd(q, k, v, o, lse, causal, softmax_scale(d), None, window, lens_t)
    assert binding.device_error() == 0
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def check(o, lse, o_ref, lse_ref, what, dtype):
    assert np.isfinite(o).all(), what
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), what
    d_o = o - o_ref
    assert (np.abs(d_o) - o_bound(o_ref, dtype)).max() <= 0, (what, float(np.abs(d_o).max()))
    if np.linalg.norm(o_ref) > 0:
        assert np.linalg.norm(d_o) / np.linalg.norm(o_ref) <= REL_L2_O, what
    if (~empty).any():
        assert np.abs(lse[~empty] - lse_ref[~empty]).max() <= MAX_ABS_LSE, what


def case(B, H, N, d, dtype, causal, window, lens, seed):
    qb, kb, vb = make_qkv(B, H, N, d, dtype, seed)
    o, lse = run_masked(qb, kb, vb, dtype, causal, window, lens)
    o_ref, lse_ref = oracle.attention(qb, kb, vb, causal, softmax_scale(d), dtype=dtype,
                                      window=window, seqlens_k=lens)
    check(o, lse, o_ref, lse_ref, (B, H, N, d, dtype, causal, window, lens), dtype)


@pytest.mark.parametrize("N", [200, 300, 513])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_padding(N, d, causal):
    case(3, 2, N, d, "bf16", causal, (-1, -1), [N, N // 2 + 3, 0], seed=300 + N)


@pytest.mark.parametrize("window,causal", [((64, -1), True), ((127, -1), True),
                                           ((128, -1), True), ((300, -1), True),
                                           ((0, -1), True), ((100, 100), False),
                                           ((0, 0), False), ((-1, 50), False),
                                           ((200, 0), False), ((5, 300), False)])
@pytest.mark.parametrize("N", [300, 700])
def test_sliding_window(window, causal, N):
    case(2, 2, N, 128, "bf16", causal, window, None, seed=400 + N)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_window_and_padding(dtype):
    case(3, 2, 641, 64, dtype, True, (150, -1), [641, 390, 77], seed=500)
    case(2, 3, 400, 128, dtype, False, (60, 20), [130, 400], seed=501)


def test_empty_everything():
    """Zero key lengths: every row is empty; a window that leaves rows past the key length
    empty."""
    case(2, 1, 260, 64, "bf16", False, (-1, -1), [0, 0], seed=502)
    case(1, 2, 300, 64, "bf16", True, (0, -1), [100], seed=503)


def test_long_window_sampled():
    """N = 8192 causal with a 1024-key window (the kernel visits ~9 K/V tiles per Q tile)."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    B, H, N, d = 1, 4, 8192, 128
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed=504)
    q, k, v = (to_device(x, "bf16") for x in (qb, kb, vb))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    binding.fa_fwd(q, k, v, o, lse, True, softmax_scale(d), None, (1024, -1))
    assert binding.device_error() == 0
    rows = sample_rows(B, H, N, 64, seed=505)
    o_ref, lse_ref = oracle.attention_rows(qb, kb, vb, rows, True, softmax_scale(d),
                                           dtype="bf16", window=(1024, -1))
    idx = [torch.from_numpy(rows[:, c]).cuda() for c in range(3)]
    check(o[idx[0], idx[2], idx[1]].double().cpu().numpy(),
          lse[idx[0], idx[1], idx[2]].double().cpu().numpy(), o_ref, lse_ref, "window 1024", "bf16")


@pytest.mark.parametrize("name", ["n8k_d128_window1k", "n8k_d128_padded"])
def test_masked_workload_sampled(name):
    """The masked workloads the benchmark times (B=2, H=16, N=8192, d=128), full size, one call
    as the bench makes it; sampled rows of every head against the fp64 oracle, plus rows past
    the shorter key length (padding) and the window's edge (sliding window)."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    w = WORKLOADS[name]
    qb, kb, vb = make_workload(w)
    q, k, v = (to_device(x, w.dtype) for x in (qb, kb, vb))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32, device=q.device)
    lens = list(w.seqlens_k) or None
    lens_t = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=q.device)
    binding.fa_fwd(q, k, v, o, lse, w.causal, w.scale, None, w.window, lens_t)
    assert binding.device_error() == 0
    rows = sample_rows(w.B, w.H, w.N, 64, seed=w.seed + 7)
    extra = [(b, h, i) for b in range(w.B) for h in (0, w.H - 1)
             for i in (1022, 1023, 1024, 1025, 4999, 5000, 5001, w.N - 1)]
    rows = np.concatenate([rows, np.array(extra, dtype=rows.dtype)])
    o_ref, lse_ref = oracle.attention_rows(qb, kb, vb, rows, w.causal, w.scale, dtype=w.dtype,
                                           window=w.window, seqlens_k=lens)
    idx = [torch.from_numpy(rows[:, c]).cuda() for c in range(3)]
    check(o[idx[0], idx[2], idx[1]].double().cpu().numpy(),
          lse[idx[0], idx[1], idx[2]].double().cpu().numpy(), o_ref, lse_ref, name, w.dtype)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_masked_bad_arguments():
    import torch

    from io_aware_attention_fa2_gb300 import binding
    lib = binding.load_library()
    q = torch.zeros(2, 128, 1, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros(2, 1, 128, device="cuda")
    lens = torch.tensor([128, 64], dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    # key lengths overlapping the LSE output
    assert lib.fa_fwd_masked(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), 2, 1, 128, 64, 0, -1, -1, lse.data_ptr(), 0.125,
                             0, st) == -5
    # misaligned key lengths
    assert lib.fa_fwd_masked(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), 2, 1, 128, 64, 0, -1, -1, lens.data_ptr() + 2,
                             0.125, 0, st) == -4
    torch.cuda.synchronize()
    assert float(o.float().abs().sum()) == 0.0
