"""Calls that overlap: forward and backward launches on several streams at once, and the
host-buffer entry points from two threads at once, each checked against the same call made
alone. The kernels keep no state between calls except the device error word, and the host
entry points serialise only their enqueueing, so every overlapped result must equal the lone one
(dQ of the backward to within one rounding: its fp32 partial sums arrive in no fixed order)."""
import threading

import numpy as np
import pytest

from gpu_util import to_device
from io_aware_attention_fa2_gb300.inputs import make_qkv, normal, round_to_bits, softmax_scale

pytestmark = pytest.mark.gpu

CASES = [(2, 4, 1000, 128, True), (1, 8, 2048, 64, False), (3, 2, 777, 128, False),
         (1, 16, 4096, 128, True)]


def _inputs(B, H, N, d, seed):
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed)
    dob = round_to_bits(normal((B, N, H, d), seed + 9), "bf16")
    return [to_device(x, "bf16") for x in (qb, kb, vb, dob)]


def _run(binding, torch, case, tensors, stream):
    B, H, N, d, causal = case
    q, k, v, do = tensors
    scale = softmax_scale(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    grads = [torch.empty_like(q) for _ in range(3)]
    ws = torch.empty(binding.bwd_workspace_size(B, H, N, d), dtype=torch.uint8,
                     device=q.device)
    binding.fa_fwd(q, k, v, o, lse, causal, scale, stream)
    binding.fa_bwd(q, k, v, o, do, lse, *grads, causal, scale, ws, stream)
    return [o, lse, *grads, ws]


def test_overlapping_streams_match_lone_calls():
    import torch

    from io_aware_attention_fa2_gb300 import binding
    inputs = [_inputs(*c[:4], seed=9700 + i) for i, c in enumerate(CASES)]
    lone = []
    for case, t in zip(CASES, inputs):
        out = _run(binding, torch, case, t, None)
        torch.cuda.synchronize()
        lone.append([x.clone() for x in out[:5]])
    streams = [torch.cuda.Stream() for _ in CASES]
    torch.cuda.synchronize()
    # enqueue everything on its own stream before waiting for any of it
    outs = []
    for case, t, st in zip(CASES, inputs, streams):
        with torch.cuda.stream(st):
            outs.append(_run(binding, torch, case, t, st))
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    for case, a, b in zip(CASES, lone, outs):
        o_a, l_a, dq_a, dk_a, dv_a = a
        o_b, l_b, dq_b, dk_b, dv_b = b[:5]
        assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b), case
        assert torch.equal(dk_a, dk_b) and torch.equal(dv_a, dv_b), case
        da, db = dq_a.double(), dq_b.double()
        assert bool((da - db).abs().le(2.0 ** -7 * da.abs() + 1e-6).all()), case


def test_host_entry_points_from_two_threads():
    """fa_fwd_host and fa_bwd_host called at the same moment from two threads (ctypes releases
    the interpreter lock during the call), each on its own stream."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    cases = [(2, 8, 2048, 128, True), (1, 6, 3000, 64, False)]
    host, ref = [], []
    for i, (B, H, N, d, causal) in enumerate(cases):
        qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed=9800 + i)
        dob = round_to_bits(normal((B, N, H, d), 9810 + i), "bf16")
        h = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
             for x in (qb, kb, vb, dob)]
        dev = [t.cuda() for t in h]
        o, lse = binding.attention_forward(*dev[:3], causal=causal)
        g = binding.attention_backward(*dev[:3], o, dev[3], lse, causal=causal)
        torch.cuda.synchronize()
        host.append(h)
        ref.append((o.cpu(), lse.cpu(), [x.cpu() for x in g]))
    results = [None, None]
    errors = []

    def work(i):
        try:
            B, H, N, d, causal = cases[i]
            st = torch.cuda.Stream()
            q, k, v, do = host[i]
            for _ in range(3):
                o, lse = binding.attention_forward(q, k, v, causal=causal, stream=st)
                g = binding.attention_backward(q, k, v, o.pin_memory(), do, lse.pin_memory(),
                                               causal=causal, stream=st)
            results[i] = (o, lse, g)
        except Exception as e:  # reported below, in the test's own thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert binding.device_error() == 0
    for (o, lse, g), (o_r, lse_r, g_r) in zip(results, ref):
        assert torch.equal(o.view(torch.int16), o_r.view(torch.int16))
        assert torch.equal(lse, lse_r)
        assert torch.equal(g[1].view(torch.int16), g_r[1].view(torch.int16))
        assert torch.equal(g[2].view(torch.int16), g_r[2].view(torch.int16))
        da, db = g[0].double(), g_r[0].double()
        assert bool((da - db).abs().le(2.0 ** -7 * db.abs() + 1e-6).all())
