"""The parity rule (``oracle.tolerance``) against facts about the storage types and the method's
own roundings (CPU only).

Half a step of bf16 / fp16 must be what the types' own spacing says (numpy's float16 spacing;
torch's bfloat16 next representable value). The element-wise forward bar must be exactly 1e-2
unless the method's two roundings can exceed it; and those bounds must hold: a simulation that
rounds P and O exactly as the method does (torch's bf16 / fp16 conversions) stays inside
half_step + u * A, and a backward that takes D from that rounded O moves dQ by no more than
``dq_allowance``.
"""
import numpy as np
import pytest

from oracle.tolerance import (MAX_ABS_O, UNIT_ROUNDOFF, dq_allowance, grad_stats, half_step,
                              o_bound, stats)


def test_half_step_fp16_matches_numpy_spacing():
    x = np.array([2.0 ** -14, 0.3, 1.0, 1.5, 3.9, 4.0, 31.9, 32.0, 1000.0, 65000.0])
    want = np.spacing(x.astype(np.float16)).astype(np.float64) / 2
    assert np.array_equal(half_step(x, "fp16"), want)


def test_half_step_bf16_matches_torch_next_value():
    torch = pytest.importorskip("torch")
    x = np.array([2.0 ** -14, 0.3, 1.0, 1.5, 3.9, 4.0, 7.99, 8.0, 1000.0, 3.0e38])
    t = torch.tensor(x, dtype=torch.float64).to(torch.bfloat16).to(torch.float64)
    nxt = torch.nextafter(t.to(torch.bfloat16), torch.tensor(float("inf"),
                                                            dtype=torch.bfloat16))
    want = (nxt.to(torch.float64) - t).numpy() / 2
    assert np.array_equal(half_step(t.numpy(), "bf16"), want)


def test_bound_is_the_stated_bar_unless_the_roundings_exceed_it():
    # bf16: half a step first exceeds 1e-2 - 1e-3 on [4, 8); fp16 on [32, 64)
    for dtype, edge in (("bf16", 4.0), ("fp16", 32.0)):
        below = np.array([0.0, 0.5, -1.0, 2.0, np.nextafter(edge, 0), -np.nextafter(edge, 0)])
        assert np.all(o_bound(below, dtype) == MAX_ABS_O)
        above = np.array([edge, -edge, 2 * edge - 0.01])
        assert np.allclose(o_bound(above, dtype), 2.0 ** -6 + 1e-3)
    # peaked attention: |O| = 3 averaging |V| entries of 3 -> half step + u * 3 + 1e-3
    assert np.isclose(o_bound(np.array([3.0]), "bf16", np.array([3.0]))[0],
                      2.0 ** -7 + 3 * 2.0 ** -8 + 1e-3)
    # typical rows (|O| small, A about 0.8) keep the stated bar
    assert o_bound(np.array([0.2]), "bf16", np.array([0.8]))[0] == MAX_ABS_O


def test_stats_flags_a_plain_miss_and_passes_rounding():
    o_ref = np.array([0.1, 5.001, -3.0])
    lse_ref = np.zeros(3)
    ok = stats(np.array([0.1099, 5.0, -3.0]), lse_ref, o_ref, lse_ref, "bf16")
    assert ok["ok"] and ok["relaxed_elements"] == 1
    bad = stats(np.array([0.1101, 5.0, -3.0]), lse_ref, o_ref, lse_ref, "bf16")
    assert not bad["ok"] and bad["max_excess_o"] > 0
    far = stats(np.array([0.1, 5.0 + 2.0 ** -5, -3.0]), lse_ref, o_ref, lse_ref, "bf16")
    assert not far["ok"]
    assert not stats(o_ref, lse_ref + 2e-3, o_ref, lse_ref, "bf16")["ok"]
    assert not stats(np.array([np.nan, 5.0, -3.0]), lse_ref, o_ref, lse_ref, "bf16")["ok"]


def _round(x, dtype):
    import torch
    t = torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.float32)
    return t.to(torch.bfloat16 if dtype == "bf16" else torch.float16).to(torch.float64).numpy()


def _case(seed, n, d, logit_scale, dtype):
    """One attention row set with P and O rounded as the method rounds them."""
    rng = np.random.default_rng(seed)
    q = _round(rng.normal(size=(n, d)) * logit_scale, dtype)
    k = _round(rng.normal(size=(n, d)), dtype)
    v = _round(rng.normal(size=(n, d)) * 2.0, dtype)
    s = q @ k.T / np.sqrt(d)
    s = s - s.max(axis=1, keepdims=True) + rng.uniform(0, 8, size=(n, 1))   # offset <= 2^8
    p = np.exp2(s * np.log2(np.e))
    w = p / p.sum(axis=1, keepdims=True)
    o_exact = w @ v
    o_rounded_p = (_round(p, dtype) @ v) / p.sum(axis=1, keepdims=True)
    o_stored = _round(o_rounded_p, dtype)
    a = w @ np.abs(v)
    return q, k, v, w, o_exact, o_stored, a


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("logit_scale", [1.0, 8.0, 30.0])
def test_forward_rounding_bound_holds_in_simulation(dtype, logit_scale):
    pytest.importorskip("torch")
    for seed in range(6):
        _, _, _, _, o_exact, o_stored, a = _case(seed, 48, 32, logit_scale, dtype)
        err = np.abs(o_stored - o_exact)
        assert (err <= half_step(o_exact, dtype) + UNIT_ROUNDOFF[dtype] * a + 1e-12).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("logit_scale", [1.0, 8.0, 30.0])
def test_dq_allowance_covers_d_from_the_stored_o(dtype, logit_scale):
    """dQ computed exactly except for D = <dO, O> taken from the stored (rounded) O moves by
    no more than dq_allowance; on unpeaked rows (logits of unit scale) a 5 % error in dQ on
    top of it is still caught."""
    pytest.importorskip("torch")
    for seed in range(6):
        q, k, v, w, o_exact, o_stored, a = _case(100 + seed, 48, 32, logit_scale, dtype)
        rng = np.random.default_rng(200 + seed)
        dout = _round(rng.normal(size=o_exact.shape), dtype)
        scale = 1.0 / np.sqrt(q.shape[1])
        dp = dout @ v.T

        def dq_with(dvec):
            return scale * (w * (dp - dvec[:, None])) @ k

        dq_exact = dq_with((dout * o_exact).sum(axis=1))
        dq_d = dq_with((dout * o_stored).sum(axis=1))
        allow = dq_allowance(scale, dtype, dout, a, w @ k)
        assert (np.abs(dq_d - dq_exact) <= allow + 1e-12).all()
        assert grad_stats(dq_d, dq_exact, dtype, "dq", allow)["ok"]
        if logit_scale == 1.0:
            assert not grad_stats(dq_d + 0.05 * dq_exact, dq_exact, dtype, "dq", allow)["ok"]
