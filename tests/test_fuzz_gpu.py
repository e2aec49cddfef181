"""Seeded random combinations of the options the other parity tests take one or two at a time:
shape (B, H, Nq, Nk, d; Nq and Nk not tile multiples), dtype, causal, a sliding window, per-batch
key lengths (empty batches included), the split-K/V part count and the scale (a negative scale
included: its path scales S before taking the row maximum). The forward of every case and the
backward of a subset go through the C ABI and are held to the common bar against the fp64
oracle; rows with no visible key must come out as O = 0 and LSE = -inf on both sides. The
element bar includes the rounding of P to the input type (u times the attention of |V|, from the
oracle): a scale of 3 / sqrt(d) or a window of a few keys makes attention peaked enough for it to
pass 1e-2 in bf16."""
import numpy as np
import pytest

import oracle
from gpu_util import (MAX_ABS_LSE, REL_L2_O, attention_aux, check_grad, dq_allowance_for,
                      o_bound, to_device)
from io_aware_attention_fa2_gb300.inputs import make_qkv, normal, round_to_bits, softmax_scale

pytestmark = pytest.mark.gpu

N_FWD = 96
N_BWD = 24


def draw(i: int, bwd: bool = False) -> dict:
    """Case i: a seeded draw of every option (the backward takes Nq = Nk and no split)."""
    rng = np.random.default_rng(4242 + 1000 * bwd + i)
    d = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["bf16", "fp16"]))
    B, H = int(rng.integers(1, 4)), int(rng.integers(1, 4))
    nq = int(rng.integers(1, 300 if bwd else 600))
    split = (not bwd) and rng.random() < 0.5
    nk = nq + (int(rng.integers(0, 700)) if split else 0)
    splits = int(rng.integers(1, 9)) if split else 1
    causal = bool(rng.random() < 0.5)
    kind = int(rng.integers(0, 4))
    left = int(rng.integers(0, 300)) if kind in (1, 3) else -1
    right = int(rng.integers(0, 300)) if kind in (2, 3) else -1
    lens = None
    if rng.random() < 0.5:
        lens = [int(rng.integers(0, nk + 1)) for _ in range(B)]
        if rng.random() < 0.3:
            lens[int(rng.integers(0, B))] = 0
    mult = float(rng.choice([1.0, 0.5, 3.0, -1.0])) if not bwd else float(rng.choice([1.0, 2.0]))
    return dict(B=B, H=H, nq=nq, nk=nk, d=d, dtype=dtype, causal=causal, window=(left, right),
                lens=lens, splits=splits, split=split,
                scale=float(np.float32(softmax_scale(d) * mult)),
                seed=7000 + 1000 * bwd + i)


def check(o, lse, o_ref, lse_ref, what, dtype, a_ref):
    assert np.isfinite(o).all(), what
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), what
    d_o = o - o_ref
    excess = (np.abs(d_o) - o_bound(o_ref, dtype, a_ref)).max()
    assert excess <= 0, (what, float(np.abs(d_o).max()), float(excess))
    if np.linalg.norm(o_ref) > 0:
        assert np.linalg.norm(d_o) / np.linalg.norm(o_ref) <= REL_L2_O, what
    if (~empty).any():
        assert np.abs(lse[~empty] - lse_ref[~empty]).max() <= MAX_ABS_LSE, what


@pytest.mark.parametrize("i", range(N_FWD))
def test_fuzz_forward(i):
    import torch

    from io_aware_attention_fa2_gb300 import binding
    c = draw(i)
    qb, kb, vb = make_qkv(c["B"], c["H"], c["nq"], c["d"], c["dtype"], c["seed"], Nk=c["nk"])
    q, k, v = (to_device(x, c["dtype"]) for x in (qb, kb, vb))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((c["B"], c["H"], c["nq"]), float("nan"), dtype=torch.float32, device="cuda")
    lens_t = None if c["lens"] is None else torch.tensor(c["lens"], dtype=torch.int32,
                                                          device="cuda")
    if c["split"]:
        binding.fa_fwd_splitkv(q, k, v, o, lse, c["causal"], c["scale"], c["splits"], None, None,
                               c["window"], lens_t)
    else:
        binding.fa_fwd(q, k, v, o, lse, c["causal"], c["scale"], None, c["window"], lens_t)
    assert binding.device_error() == 0
    o_ref, lse_ref = oracle.attention(qb, kb, vb, c["causal"], c["scale"], dtype=c["dtype"],
                                      window=c["window"], seqlens_k=c["lens"])
    a_ref, _ = attention_aux(qb, kb, vb, c["causal"], c["scale"], c["dtype"], None, c["window"],
                             c["lens"])
    check(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, c, c["dtype"],
          a_ref)


@pytest.mark.parametrize("i", range(N_BWD))
def test_fuzz_backward(i):
    import torch

    from io_aware_attention_fa2_gb300 import binding
    c = draw(i, bwd=True)
    B, H, N, d, dtype = c["B"], c["H"], c["nq"], c["d"], c["dtype"]
    qb, kb, vb = make_qkv(B, H, N, d, dtype, c["seed"])
    dob = round_to_bits(normal((B, N, H, d), c["seed"] + 1), dtype)
    q, k, v, do = (to_device(x, dtype) for x in (qb, kb, vb, dob))
    lens_t = None if c["lens"] is None else torch.tensor(c["lens"], dtype=torch.int32,
                                                          device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    binding.fa_fwd(q, k, v, o, lse, c["causal"], c["scale"], None, c["window"], lens_t)
    grads = [torch.full_like(q, float("nan")) for _ in range(3)]
    binding.fa_bwd(q, k, v, o, do, lse, *grads, c["causal"], c["scale"], None, None, c["window"],
                   lens_t)
    assert binding.device_error() == 0
    refs = oracle.attention_bwd(qb, kb, vb, dob, c["causal"], c["scale"], dtype=dtype,
                                window=c["window"], seqlens_k=c["lens"])
    allow = dq_allowance_for(qb, kb, vb, dob, c["causal"], c["scale"], dtype,
                             window=c["window"], seqlens_k=c["lens"])
    for j, (name, g, r) in enumerate(zip(("dq", "dk", "dv"), grads, refs)):
        check_grad(name, g.double().cpu().numpy(), r, dtype, c, allow if j == 0 else None)


N_HOST = 16


def host_tensor(bits: np.ndarray, dtype: str):
    """A CPU tensor (pinned) of the bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16).pin_memory()


@pytest.mark.parametrize("i", range(N_HOST))
def test_fuzz_host_forward(i):
    """The host-buffer forward (copies in and out around the kernels, head groups overlapped)."""
    import torch

    from io_aware_attention_fa2_gb300 import attention_forward
    c = draw(100 + i, bwd=True)   # queries and keys share N on the host-buffer path
    qb, kb, vb = make_qkv(c["B"], c["H"], c["nq"], c["d"], c["dtype"], c["seed"])
    lens_t = None if c["lens"] is None else torch.tensor(c["lens"], dtype=torch.int32)
    o, lse = attention_forward(*(host_tensor(x, c["dtype"]) for x in (qb, kb, vb)),
                               causal=c["causal"], scale=c["scale"], window=c["window"],
                               seqlens_k=lens_t)
    assert not o.is_cuda and not lse.is_cuda
    o_ref, lse_ref = oracle.attention(qb, kb, vb, c["causal"], c["scale"], dtype=c["dtype"],
                                      window=c["window"], seqlens_k=c["lens"])
    a_ref, _ = attention_aux(qb, kb, vb, c["causal"], c["scale"], c["dtype"], None, c["window"],
                             c["lens"])
    check(o.double().numpy(), lse.double().numpy(), o_ref, lse_ref, c, c["dtype"], a_ref)


@pytest.mark.parametrize("i", range(N_HOST // 2))
def test_fuzz_host_backward(i):
    """The host-buffer backward on the host-buffer forward's O and LSE."""
    import torch

    from io_aware_attention_fa2_gb300 import attention_backward, attention_forward
    c = draw(200 + i, bwd=True)
    B, H, N, d, dtype = c["B"], c["H"], c["nq"], c["d"], c["dtype"]
    qb, kb, vb = make_qkv(B, H, N, d, dtype, c["seed"])
    dob = round_to_bits(normal((B, N, H, d), c["seed"] + 1), dtype)
    q, k, v, do = (host_tensor(x, dtype) for x in (qb, kb, vb, dob))
    lens_t = None if c["lens"] is None else torch.tensor(c["lens"], dtype=torch.int32)
    kw = dict(causal=c["causal"], scale=c["scale"], window=c["window"], seqlens_k=lens_t)
    o, lse = attention_forward(q, k, v, **kw)
    grads = attention_backward(q, k, v, o, do, lse, **kw)
    refs = oracle.attention_bwd(qb, kb, vb, dob, c["causal"], c["scale"], dtype=dtype,
                                window=c["window"], seqlens_k=c["lens"])
    allow = dq_allowance_for(qb, kb, vb, dob, c["causal"], c["scale"], dtype,
                             window=c["window"], seqlens_k=c["lens"])
    for j, (name, g, r) in enumerate(zip(("dq", "dk", "dv"), grads, refs)):
        assert not g.is_cuda
        check_grad(name, g.double().numpy(), r, dtype, c, allow if j == 0 else None)
