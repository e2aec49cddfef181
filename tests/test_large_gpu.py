"""Maximum sizes: tensors of more than 2^31 elements (byte offsets past 4 GiB), through the
forward, the backward and the split-K/V forward, checked on sampled heads against the oracle.

The big tensors are filled on the device with a seeded normal filler; the sampled (b, h) heads
are then overwritten with the seeded inputs the oracle also gets, so the oracle needs only those
heads (attention of one head depends on that head alone). The samples sit at the start, the
middle, just below and just above element 2^31 and at the very end of the tensors, so an index
computed in 32 bits would read or write the wrong head. Outputs start as NaN: a row that is not
written fails.
"""
import numpy as np
import pytest

import oracle
from gpu_util import (MAX_ABS_LSE, REL_L2_O, check_grad, dq_allowance_for, o_bound,
                      to_device)
from io_aware_attention_fa2_gb300.inputs import make_qkv, normal, round_to_bits, softmax_scale

pytestmark = pytest.mark.gpu


def _filled(shape, seed):
    import torch
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda", dtype=torch.bfloat16)


def _plant(big, b, h, bits):
    big[b, :, h, :] = to_device(bits, "bf16")[0, :, 0, :]


def _heads_past_2_31(B, N, H, d):
    """(b, h) samples: first, middle, last below element 2^31, first at or above it, last."""
    per_b = N * H * d
    b_cross = (1 << 31) // per_b
    assert b_cross * per_b == 1 << 31 and b_cross < B - 1, "shape must straddle 2^31 at a batch"
    return [(0, 0), (B // 2, H // 2 - 3), (b_cross - 1, H - 1), (b_cross, 0), (B - 1, H - 1)]


def _check(o, lse, o_ref, lse_ref, what):
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    d_o = o - o_ref
    assert (np.abs(d_o) - o_bound(o_ref, "bf16")).max() <= 0, (what, float(np.abs(d_o).max()))
    assert np.linalg.norm(d_o) / np.linalg.norm(o_ref) <= REL_L2_O, what
    assert np.abs(lse - lse_ref).max() <= MAX_ABS_LSE, what


def test_forward_and_backward_past_2_31_elements():
    """B=1152, H=64, N=256, d=128 bf16 (2.4 G elements, 4.8 GB per tensor), causal: forward O
    and LSE, then dQ, dK, dV of the same attention, on five sampled heads."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    B, H, N, d = 1152, 64, 256, 128
    assert B * N * H * d > 1 << 31
    scale = softmax_scale(d)
    heads = _heads_past_2_31(B, N, H, d)
    q, k, v, do = (_filled((B, N, H, d), 9100 + i) for i in range(4))
    small = {}
    for n, (b, h) in enumerate(heads):
        qb, kb, vb = make_qkv(1, 1, N, d, "bf16", seed=9200 + n)
        dob = round_to_bits(normal((1, N, 1, d), 9300 + n), "bf16")
        for big, bits in ((q, qb), (k, kb), (v, vb), (do, dob)):
            _plant(big, b, h, bits)
        small[(b, h)] = (qb, kb, vb, dob)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    binding.fa_fwd(q, k, v, o, lse, True, scale)
    assert binding.device_error() == 0
    for (b, h), (qb, kb, vb, _) in small.items():
        o_ref, lse_ref = oracle.attention(qb, kb, vb, True, scale, dtype="bf16")
        got_o = o[b, :, h, :].double().cpu().numpy()[None, :, None, :]
        got_l = lse[b, h, :].double().cpu().numpy()[None, None, :]
        _check(got_o, got_l, o_ref, lse_ref, ("fwd", b, h))

    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    binding.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, True, scale)
    assert binding.device_error() == 0
    for (b, h), (qb, kb, vb, dob) in small.items():
        refs = oracle.attention_bwd(qb, kb, vb, dob, True, scale, dtype="bf16")
        allow = dq_allowance_for(qb, kb, vb, dob, True, scale, "bf16")
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
            got = g[b, :, h, :].double().cpu().numpy()[None, :, None, :]
            check_grad(name, got, r, "bf16", ("past 2^31", b, h),
                       allow if name == "dq" else None)
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()


def test_splitkv_keys_past_2_31_elements():
    """One query against 65,536 keys, B=16, H=20, d=128 bf16 (K and V 2.7 G elements each),
    split over K/V parts and merged, on five sampled heads (the keys of the fourth and fifth,
    and the later keys of the third, lie past element 2^31)."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    B, H, Nk, d = 16, 20, 65536, 128
    scale = softmax_scale(d)
    b_cross = ((1 << 31) + Nk * H * d - 1) // (Nk * H * d)   # first batch past element 2^31
    heads = [(0, 0), (3, 17), (b_cross - 1, H - 1), (b_cross, 0), (B - 1, H - 1)]
    assert B * Nk * H * d > 1 << 31 and b_cross < B - 1
    q = _filled((B, 1, H, d), 9400)
    k, v = (_filled((B, Nk, H, d), 9401 + i) for i in range(2))
    small = {}
    for n, (b, h) in enumerate(heads):
        qb, kb, vb = make_qkv(1, 1, 1, d, "bf16", seed=9500 + n, Nk=Nk)
        for big, bits in ((q, qb), (k, kb), (v, vb)):
            _plant(big, b, h, bits)
        small[(b, h)] = (qb, kb, vb)
    splits = binding.splitkv_num_splits(B, H, 1, Nk)
    assert splits > 1
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, 1), float("nan"), dtype=torch.float32, device="cuda")
    binding.fa_fwd_splitkv(q, k, v, o, lse, True, scale, splits)
    assert binding.device_error() == 0
    for (b, h), (qb, kb, vb) in small.items():
        o_ref, lse_ref = oracle.attention(qb, kb, vb, True, scale, dtype="bf16")
        got_o = o[b, :, h, :].double().cpu().numpy()[None, :, None, :]
        got_l = lse[b, h, :].double().cpu().numpy()[None, None, :]
        _check(got_o, got_l, o_ref, lse_ref, ("splitkv", b, h, splits))
    del q, k, v, o, lse
    torch.cuda.empty_cache()
