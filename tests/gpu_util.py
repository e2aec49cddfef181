"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on bit-exact copies of
the seeded inputs, and compare with the oracle.

The bar is one rule for every test (``oracle.tolerance``): max |dO| <= 1e-2 element-wise,
||dO||_2 / ||O_ref||_2 <= 5e-3, max |dLSE| <= 1e-3, against the oracle's unrounded fp64
values; only where half a step of the output type at |O_ref| is itself above 1e-2 (|O_ref| >= 4
in bf16, >= 32 in fp16) is the element's bar 1e-2 plus that half step.
"""
from __future__ import annotations

import numpy as np

from oracle.tolerance import (MAX_ABS_LSE, MAX_ABS_O, REL_L2_O, attention_aux,
                              dq_allowance_for, grad_stats, half_step, o_bound, stats)

__all__ = ["MAX_ABS_O", "REL_L2_O", "MAX_ABS_LSE", "half_step", "o_bound", "to_device",
           "run_gpu", "assert_close", "check_grad", "ERROR_LOG", "attention_aux",
           "dq_allowance_for"]

# Every comparison made through assert_close / check_grad, in order: the measured errors behind
# the bars. conftest.py writes it to the file named by FA_ERROR_LOG at the end of the session.
ERROR_LOG: list[dict] = []


def to_device(bits: np.ndarray, dtype: str):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    t = t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.cuda()


def run_gpu(qb, kb, vb, dtype: str, causal: bool, scale: float, check_error: bool = True):
    """fa_fwd on the GPU. Returns (o float64 [B,N,H,d], lse float64 [B,H,N]) as numpy."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    q, k, v = (to_device(x, dtype) for x in (qb, kb, vb))
    B, N, H, d = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    binding.fa_fwd(q, k, v, o, lse, causal, scale)
    if check_error:
        assert binding.device_error() == 0, "a kernel wait ran out"
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def assert_close(o, lse, o_ref, lse_ref, what: str, dtype: str, a_ref=None):
    """Assert the bar of ``oracle.tolerance`` for an output stored in ``dtype`` (``a_ref``: the
    oracle's attention of |V| on the same rows, or None for the stricter bar without it)."""
    st = stats(o, lse, o_ref, lse_ref, dtype, a_ref)
    ERROR_LOG.append({"what": str(what), "dtype": dtype, **st})
    assert st["finite"], "non-finite output %s" % what
    assert st["max_excess_o"] <= 0.0, (what, st)
    assert st["rel_l2_o"] <= REL_L2_O, (what, st)
    assert st["max_abs_lse"] <= MAX_ABS_LSE, (what, st)
    return st


def check_grad(name: str, g, r, dtype: str, what, allowance=None) -> dict:
    """Assert the backward bar of ``oracle.tolerance`` for one gradient (dq, dk or dv);
    ``allowance``: dQ's allowance for D taken from the stored O (``dq_allowance_for``)."""
    st = grad_stats(g, r, dtype, name, allowance)
    ERROR_LOG.append({"what": str(what), "grad": name, "dtype": dtype, **st})
    assert st["ok"], (name, what, st)
    return st
