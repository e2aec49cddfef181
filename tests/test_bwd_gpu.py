"""Parity of the backward (fa_bwd) with the fp64 oracle's gradients.

The GPU forward provides O and LSE (as a user would run it); the oracle differentiates the exact
definition on the same bf16/fp16 inputs. The bar (``oracle.tolerance.grad_bars``) follows from
the arithmetic: with u the unit roundoff of the input type (2^-8 bf16, 2^-11 fp16), P and dS
are rounded to the input type before their products, D uses the rounded O and the outputs are
rounded, so each gradient is held to a relative L2 error of 2u and a largest element error of
6u of its largest element. Where the exact gradient vanishes (dQ and dK with a single key), the
computed one must stay below 1e-3.
"""
import numpy as np
import pytest

import oracle
from gpu_util import check_grad, dq_allowance_for, to_device
from io_aware_attention_fa2_gb300.inputs import (WORKLOADS, make_qkv, make_workload, normal,
                                                 round_to_bits, softmax_scale)

pytestmark = pytest.mark.gpu

def run_case(B, H, N, d, dtype, causal, seed):
    import torch

    from io_aware_attention_fa2_gb300 import binding
    qb, kb, vb = make_qkv(B, H, N, d, dtype, seed)
    dob = round_to_bits(normal((B, N, H, d), seed + 9), dtype)
    q, k, v, do = (to_device(x, dtype) for x in (qb, kb, vb, dob))
    scale = softmax_scale(d)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    binding.fa_fwd(q, k, v, o, lse, causal, scale)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    binding.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, causal, scale)
    assert binding.device_error() == 0
    got = [t.double().cpu().numpy() for t in (dq, dk, dv)]
    ref = oracle.attention_bwd(qb, kb, vb, dob, causal, scale, dtype=dtype)
    allow = dq_allowance_for(qb, kb, vb, dob, causal, scale, dtype)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        check_grad(name, g, r, dtype, (B, H, N, d, dtype, causal),
                   allow if name == "dq" else None)


@pytest.mark.parametrize("N", [1, 17, 128, 200, 257])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_shapes(N, d, causal):
    run_case(2, 2, N, d, "bf16", causal, seed=900 + N + d)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_fp16(causal):
    run_case(1, 3, 300, 128, "fp16", causal, seed=990)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_longer(causal):
    run_case(1, 4, 1024, 128, "bf16", causal, seed=991)


@pytest.mark.parametrize("name", ["n1k_d128", "n1k_d64", "n1k_d64_causal"])
def test_bwd_workload_every_element(name):
    """The N = 1K workloads (B=2 H=16 d=128 and B=4 H=16 d=64, the latter causal and not) with
    the bench's upstream gradient, one fa_bwd call as the bench launches it; every element of
    dQ, dK and dV against the full fp64 gradients."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    w = WORKLOADS[name]
    qb, kb, vb = make_workload(w)
    dob = round_to_bits(normal(qb.shape, w.seed + 9), w.dtype)
    q, k, v, do = (to_device(x, w.dtype) for x in (qb, kb, vb, dob))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, device="cuda")
    binding.fa_fwd(q, k, v, o, lse, w.causal, w.scale)
    grads = [torch.full_like(q, float("nan")) for _ in range(3)]
    binding.fa_bwd(q, k, v, o, do, lse, *grads, w.causal, w.scale)
    assert binding.device_error() == 0
    ref = oracle.attention_bwd(qb, kb, vb, dob, w.causal, w.scale, dtype=w.dtype)
    allow = dq_allowance_for(qb, kb, vb, dob, w.causal, w.scale, w.dtype)
    for name_g, g, r in zip(("dq", "dk", "dv"), grads, ref):
        check_grad(name_g, g.double().cpu().numpy(), r, w.dtype, name,
                   allow if name_g == "dq" else None)


def test_bwd_bad_arguments():
    import torch

    from io_aware_attention_fa2_gb300 import binding
    q = torch.zeros(1, 128, 1, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 128, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.FaError) as e:
        binding.fa_bwd(q, q, q, q, q, lse, torch.empty_like(q), torch.empty_like(q),
                       torch.empty_like(q), False, 0.125, small)
    assert e.value.code == -11
    with pytest.raises(binding.FaError) as e:
        binding.fa_bwd(q, q, q, q, q, lse, q, torch.empty_like(q), torch.empty_like(q), False,
                       0.125)
    assert e.value.code == -5


ALL_HEADS = "all"


@pytest.mark.parametrize("name,heads", [("n8k_d128_causal", ALL_HEADS),
                                        ("n8k_d128", [(1, 7)]),
                                        ("n2000_d128_fp16_stress", [(0, 0), (15, 31)]),
                                        ("n1k_d64_causal", [(3, 15)])])
def test_bwd_full_size_sampled(name, heads):
    """Full-size workloads (the benchmarked B=2, H=16, N=8192, d=128 bf16 shape -- every one of
    its 32 heads --, the fp16 stress shape with its large logits, d=64) with the bench's
    upstream gradient, one fa_bwd call as the bench launches it; dQ, dK, dV compared on sampled
    positions against the sampled fp64 oracle: both sides of every 128-row tile edge near the
    start, middle and end (the causal diagonal of a key block runs through its own Q tile),
    the last row, and seeded ones."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    w = WORKLOADS[name]
    if heads == ALL_HEADS:
        heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    qb, kb, vb = make_workload(w)
    dob = round_to_bits(normal(qb.shape, w.seed + 9), w.dtype)
    q, k, v, do = (to_device(x, w.dtype) for x in (qb, kb, vb, dob))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, device="cuda")
    binding.fa_fwd(q, k, v, o, lse, w.causal, w.scale)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    binding.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, w.causal, w.scale)
    assert binding.device_error() == 0
    mid = (w.N // 2) // 128 * 128
    edges = [0, 1, 127, 128, 129, 255, 256, mid - 1, mid, mid + 127, w.N - 129, w.N - 128,
             w.N - 1]
    pos = np.unique(np.concatenate([[p for p in edges if 0 <= p < w.N],
                                    np.random.default_rng(w.seed + 17).integers(0, w.N, 8)]))
    ref = oracle.attention_bwd_sampled(qb, kb, vb, dob, w.causal, w.scale, heads, pos, pos,
                                       dtype=w.dtype)
    rows = [(b, h, i) for b, h in heads for i in pos]
    allow = dq_allowance_for(qb, kb, vb, dob, w.causal, w.scale, w.dtype, rows)
    allow = allow.reshape(len(heads), len(pos), -1)
    sel = torch.from_numpy(pos).cuda()
    for t, (b, h) in enumerate(heads):
        for name_g, g_all, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            g = g_all[b, sel, h].double().cpu().numpy()
            check_grad(name_g, g, r[t], w.dtype, (name, b, h),
                       allow[t] if name_g == "dq" else None)


@pytest.mark.parametrize("B,H,N,d,causal,pinned", [
    (1, 4, 200, 64, True, True), (3, 4, 1000, 128, False, True),
    (2, 16, 8192, 128, True, True),     # several head groups
    (3, 11, 4096, 64, False, False)])   # uneven groups, pageable host memory
def test_bwd_host_entry_matches_device_path(B, H, N, d, causal, pinned):
    """fa_bwd_host (host buffers, head groups packed by pitched copies, copies overlapping the
    kernels) gives the device path's gradients: dK and dV exactly (each is written once by one
    CTA); dQ to within one rounding of the output type, since its fp32 partial sums arrive from
    the key blocks' CTAs in no fixed order."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed=8500 + B + N)
    dob = round_to_bits(normal((B, N, H, d), 8600 + N), "bf16")
    host = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) for x in (qb, kb, vb, dob)]
    dev = [t.cuda() for t in host]
    o, lse = binding.attention_forward(*dev[:3], causal=causal)
    ins = host[:3] + [o.cpu(), host[3], lse.cpu()]
    if pinned:
        ins = [t.pin_memory() for t in ins]
    g_h = binding.attention_backward(*ins, causal=causal)
    g_d = binding.attention_backward(*dev[:3], o, dev[3], lse, causal=causal)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    assert all(not t.is_cuda for t in g_h)
    for name, a, b in zip(("dk", "dv"), g_h[1:], g_d[1:]):
        assert torch.equal(a.view(torch.int16), b.cpu().view(torch.int16)), name
    dq_h, dq_d = g_h[0].double(), g_d[0].cpu().double()
    assert torch.isfinite(dq_h).all()
    assert (dq_h - dq_d).abs().le(2.0 ** -7 * dq_d.abs() + 1e-6).all()


def test_bwd_host_workspace_with_and_without_headroom():
    """fa_bwd_host with exactly fa_bwd_workspace_size bytes (3 head groups whose own parts would
    need padding to 16 bytes, so they run one after another in the start of it) and with 128
    bytes more (each group in a part of its own, the groups' kernels overlapping): both give the
    device path's gradients."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    B, H, N, d, causal = 1, 6, 4097, 128, True
    assert (B * (H // 3) * N) % 4 != 0   # a group's part is not a multiple of 16 bytes
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed=8700)
    dob = round_to_bits(normal((B, N, H, d), 8701), "bf16")
    host = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
            for x in (qb, kb, vb, dob)]
    dev = [t.cuda() for t in host]
    o, lse = binding.attention_forward(*dev[:3], causal=causal)
    g_d = [t.cpu() for t in binding.attention_backward(*dev[:3], o, dev[3], lse, causal=causal)]
    o_h, lse_h = o.cpu().pin_memory(), lse.cpu().pin_memory()
    lib = binding.load_library()
    scale = softmax_scale(d)
    need = binding.bwd_workspace_size(B, H, N, d)
    for extra in (0, 128):
        outs = [torch.full_like(host[0], float("nan")).pin_memory() for _ in range(3)]
        bufs = [torch.empty_like(dev[0]) for _ in range(8)]
        ld = torch.empty(B, H, N, device="cuda")
        ws = torch.empty(need + extra, dtype=torch.uint8, device="cuda")
        st = torch.cuda.current_stream()
        rc = lib.fa_bwd_host(*(t.data_ptr() for t in (*host[:3], o_h, host[3], lse_h, *outs)),
                             *(t.data_ptr() for t in bufs[:5]), ld.data_ptr(),
                             *(t.data_ptr() for t in bufs[5:]), ws.data_ptr(), need + extra,
                             B, H, N, d, int(causal), scale, 0, st.cuda_stream)
        assert rc == 0, binding.error_string(rc)
        st.synchronize()
        assert binding.device_error() == 0
        for name, a, b in zip(("dk", "dv"), outs[1:], g_d[1:]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (extra, name)
        dq_h, dq_d = outs[0].double(), g_d[0].double()
        assert torch.isfinite(dq_h).all(), extra
        assert (dq_h - dq_d).abs().le(2.0 ** -7 * dq_d.abs() + 1e-6).all(), extra


def run_masked_case(B, H, N, d, causal, window, lens, seed):
    """fa_fwd / fa_bwd with the window and key-length masks against the oracle's gradients of
    the same masked attention."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed)
    dob = round_to_bits(normal((B, N, H, d), seed + 9), "bf16")
    q, k, v, do = (to_device(x, "bf16") for x in (qb, kb, vb, dob))
    scale = softmax_scale(d)
    lens_t = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    binding.fa_fwd(q, k, v, o, lse, causal, scale, None, window, lens_t)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    binding.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, causal, scale, None, None, window, lens_t)
    assert binding.device_error() == 0
    got = [t.double().cpu().numpy() for t in (dq, dk, dv)]
    ref = oracle.attention_bwd(qb, kb, vb, dob, causal, scale, dtype="bf16", window=window,
                               seqlens_k=lens)
    allow = dq_allowance_for(qb, kb, vb, dob, causal, scale, "bf16", window=window,
                             seqlens_k=lens)
    what = (B, H, N, d, causal, window, lens)
    # keys past a batch's key length have no query, and a batch with no key has no gradient
    # at all: exactly zero on the GPU as well
    for b, n in enumerate(lens or []):
        assert not got[1][b, n:].any() and not got[2][b, n:].any(), what
        if n == 0:
            assert not got[0][b].any(), what
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        check_grad(name, g, r, "bf16", what, allow if name == "dq" else None)


MASKS = [((64, 0), None), ((100, 30), None), ((0, 0), None), ((-1, -1), "third"),
         ((50, -1), "half_and_empty"), ((300, 200), "ragged")]


@pytest.mark.parametrize("N", [200, 513])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window,lens", MASKS, ids=[str(m) for m in MASKS])
def test_bwd_masks(N, d, causal, window, lens):
    """Sliding windows (one-sided, two-sided, the diagonal alone), key lengths (one batch with
    no key at all, lengths that are not tile multiples), with and without causal."""
    lens = {None: None, "third": [N, N // 3], "half_and_empty": [N // 2, 0],
            "ragged": [N - 1, 129]}[lens]
    run_masked_case(2, 2, N, d, causal, window, lens, seed=9900 + N + d)


@pytest.mark.parametrize("name,heads", [("n8k_d128_window1k", [(0, 5), (1, 14)]),
                                        ("n8k_d128_padded", [(0, 2), (1, 9)])])
def test_bwd_masked_full_size_sampled(name, heads):
    """The masked workloads at full size (B=2, H=16, N=8192, d=128 bf16: a causal 1024-key
    window; key lengths 8192 and 5000), one fa_bwd call with the bench's upstream gradient;
    sampled positions (tile edges, the window edge, the key-length edge, the last row) against
    the sampled oracle with the same masks."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    w = WORKLOADS[name]
    qb, kb, vb = make_workload(w)
    dob = round_to_bits(normal(qb.shape, w.seed + 9), w.dtype)
    q, k, v, do = (to_device(x, w.dtype) for x in (qb, kb, vb, dob))
    lens = list(w.seqlens_k) if w.seqlens_k else None
    lens_t = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, device="cuda")
    binding.fa_fwd(q, k, v, o, lse, w.causal, w.scale, None, w.window, lens_t)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    binding.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, w.causal, w.scale, None, None, w.window,
                   lens_t)
    assert binding.device_error() == 0
    pos = np.unique(np.concatenate([[0, 1, 127, 128, 1023, 1024, 1025, 4999, 5000, 5001,
                                     w.N // 2, w.N - 1],
                                    np.random.default_rng(w.seed + 17).integers(0, w.N, 8)]))
    ref = oracle.attention_bwd_sampled(qb, kb, vb, dob, w.causal, w.scale, heads, pos, pos,
                                       dtype=w.dtype, window=w.window, seqlens_k=lens)
    rows = [(b, h, i) for b, h in heads for i in pos]
    allow = dq_allowance_for(qb, kb, vb, dob, w.causal, w.scale, w.dtype, rows, w.window, lens)
    allow = allow.reshape(len(heads), len(pos), -1)
    sel = torch.from_numpy(pos).cuda()
    for t, (b, h) in enumerate(heads):
        for name_g, g_all, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            g = g_all[b, sel, h].double().cpu().numpy()
            if lens and name_g != "dq":
                assert not g[pos >= lens[b]].any(), (name, b, h, name_g)
            check_grad(name_g, g, r[t], w.dtype, (name, b, h),
                       allow[t] if name_g == "dq" else None)


def test_bwd_masked_host_path_matches_device_path():
    """attention_backward with host tensors and masks (copies, fa_bwd_masked, copies back)
    gives the device path's gradients."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    B, H, N, d = 2, 3, 700, 128
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed=9950)
    dob = round_to_bits(normal((B, N, H, d), 9951), "bf16")
    host = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) for x in (qb, kb, vb, dob)]
    dev = [t.cuda() for t in host]
    window, lens = (200, 0), [700, 333]
    lens_t = torch.tensor(lens, dtype=torch.int32)
    o, lse = binding.attention_forward(*dev[:3], causal=True, window=window,
                                       seqlens_k=lens_t.cuda())
    g_d = binding.attention_backward(*dev[:3], o, dev[3], lse, causal=True, window=window,
                                     seqlens_k=lens_t.cuda())
    g_h = binding.attention_backward(*host[:3], o.cpu(), host[3], lse.cpu(), causal=True,
                                     window=window, seqlens_k=lens_t)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    for a, b in zip(g_h[1:], g_d[1:]):
        assert torch.equal(a.view(torch.int16), b.cpu().view(torch.int16))
    da, db = g_h[0].double(), g_d[0].cpu().double()
    assert bool((da - db).abs().le(2.0 ** -7 * db.abs() + 1e-6).all())


def test_bwd_partial_dispatch_group():
    """B=1, H=11, N=8192, d=128: the backward's dispatch groups hold 8 heads (their Q, dO and dQ
    partial sums within 64 MiB of L2), so the last group has 3; heads of both groups checked on
    sampled positions against the sampled oracle."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    B, H, N, d = 1, 11, 8192, 128
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed=9960)
    dob = round_to_bits(normal((B, N, H, d), 9961), "bf16")
    q, k, v, do = (to_device(x, "bf16") for x in (qb, kb, vb, dob))
    scale = softmax_scale(d)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    binding.fa_fwd(q, k, v, o, lse, True, scale)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    binding.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, True, scale)
    assert binding.device_error() == 0
    heads = [(0, 0), (0, 7), (0, 8), (0, 10)]
    pos = np.array([0, 1, 127, 128, 4095, 4096, 8063, 8064, 8191])
    ref = oracle.attention_bwd_sampled(qb, kb, vb, dob, True, scale, heads, pos, pos,
                                       dtype="bf16")
    rows = [(b, h, i) for b, h in heads for i in pos]
    allow = dq_allowance_for(qb, kb, vb, dob, True, scale, "bf16", rows)
    allow = allow.reshape(len(heads), len(pos), -1)
    sel = torch.from_numpy(pos).cuda()
    for t, (b, h) in enumerate(heads):
        for name, g_all, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            g = g_all[b, sel, h].double().cpu().numpy()
            check_grad(name, g, r[t], "bf16", ("H=11 groups", h),
                       allow[t] if name == "dq" else None)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_masks_fp16(causal):
    """The masked backward in fp16 (window and key lengths together)."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    B, H, N, d = 2, 3, 333, 128
    qb, kb, vb = make_qkv(B, H, N, d, "fp16", seed=9970)
    dob = round_to_bits(normal((B, N, H, d), 9971), "fp16")
    q, k, v, do = (to_device(x, "fp16") for x in (qb, kb, vb, dob))
    scale = softmax_scale(d)
    window, lens = (90, 40), [333, 150]
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    binding.fa_fwd(q, k, v, o, lse, causal, scale, None, window, lens_t)
    grads = [torch.full_like(q, float("nan")) for _ in range(3)]
    binding.fa_bwd(q, k, v, o, do, lse, *grads, causal, scale, None, None, window, lens_t)
    assert binding.device_error() == 0
    ref = oracle.attention_bwd(qb, kb, vb, dob, causal, scale, dtype="fp16", window=window,
                               seqlens_k=lens)
    allow = dq_allowance_for(qb, kb, vb, dob, causal, scale, "fp16", window=window,
                             seqlens_k=lens)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        check_grad(name, g.double().cpu().numpy(), r, "fp16", ("masked fp16", causal),
                   allow if name == "dq" else None)


@pytest.mark.parametrize("scale", [0.0, -0.09, 1.0])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_scale_values(scale, causal):
    """Scales other than 1/sqrt(d): zero (uniform P; dQ and dK vanish), negative, and 1 (large
    logits). The forward's LSE carries the scale into P; dK and dQ take it at the end."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    B, H, N, d = 1, 3, 300, 64
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed=9990)
    dob = round_to_bits(normal((B, N, H, d), 9991), "bf16")
    q, k, v, do = (to_device(x, "bf16") for x in (qb, kb, vb, dob))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    binding.fa_fwd(q, k, v, o, lse, causal, scale)
    grads = [torch.full_like(q, float("nan")) for _ in range(3)]
    binding.fa_bwd(q, k, v, o, do, lse, *grads, causal, scale)
    assert binding.device_error() == 0
    ref = oracle.attention_bwd(qb, kb, vb, dob, causal, scale, dtype="bf16")
    allow = dq_allowance_for(qb, kb, vb, dob, causal, scale, "bf16")
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        check_grad(name, g.double().cpu().numpy(), r, "bf16", ("scale", scale, causal),
                   allow if name == "dq" else None)
