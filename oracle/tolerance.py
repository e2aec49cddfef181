"""The parity bar between the kernel's output and the fp64 oracle, as one rule for every check.

TEST INFRASTRUCTURE (part of the oracle package; see ``oracle/__init__.py``). The tests and
the benchmark's parity check (outside its timed region) apply this rule; the product never
imports it.

The stated bar for the attention forward, against the oracle's unrounded fp64 O and LSE:
    max |O - O_ref| <= 1e-2,   ||O - O_ref||_2 / ||O_ref||_2 <= 5e-3,   max |LSE - LSE_ref| <= 1e-3.

Two roundings belong to the method itself and no implementation of it avoids them: P is
rounded to the 16-bit input type before the P V product, and O is stored in that type (the
pages keep Q, K, V, O in half precision and feed P to the second matrix product). With u the
input type's unit roundoff (2^-8 bf16, 2^-11 fp16), the first moves element (i, c) of O by
at most u * A_ic, where A_ic = sum_j w_ij |v_jc| is the same attention applied to |V| (w the
softmax weights); the second by half a step of the output type at |O_ic|. Where those two
alone can exceed 1e-2 -- attention peaked on a few keys with large |V| entries, or |O| >= 4 in
bf16 (>= 32 in fp16), where half a step is itself above 1e-2 -- the element-wise bar is their
bound plus 1e-3 for the fp32 arithmetic:
    |O_ic - O_ref,ic| <= max(1e-2, half_step(O_ref,ic) + u * A_ic + 1e-3).
Everywhere else this is exactly the stated 1e-2. A is computed by the oracle (``attention``
on the same Q, K and the magnitudes of V); a check that does not compute it takes A = 0,
which only makes the bar stricter.

The relative L2 bar and the LSE bar are applied unchanged (LSE is fp32, far finer than 1e-3).
"""
from __future__ import annotations

import numpy as np

MAX_ABS_O = 1e-2
REL_L2_O = 5e-3
MAX_ABS_LSE = 1e-3
FP32_SLACK = 1e-3
UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}

_SIGNIFICANT_BITS = {"bf16": 8, "fp16": 11}


def half_step(x: np.ndarray, dtype: str) -> np.ndarray:
    """Half the spacing of representable ``dtype`` numbers in the binade of |x| (normal range;
    values below 2^-14 are taken at 2^-14, where the step is far below every bar here)."""
    bits = _SIGNIFICANT_BITS[dtype]
    _, e = np.frexp(np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -14))
    return np.ldexp(0.5, e - bits)       # |x| in [2^(e-1), 2^e): step 2^(e-1-(bits-1))


def o_bound(o_ref: np.ndarray, dtype: str, a_ref: np.ndarray | None = None) -> np.ndarray:
    """Element-wise bar on |O - O_ref| for an output stored in ``dtype``: the larger of 1e-2
    and the bound of the method's own roundings (``a_ref`` = the attention of |V|, or None
    for 0)."""
    r = half_step(o_ref, dtype) + FP32_SLACK
    if a_ref is not None:
        r = r + UNIT_ROUNDOFF[dtype] * np.abs(np.asarray(a_ref, dtype=np.float64))
    return np.maximum(MAX_ABS_O, r)


def magnitude_bits(bits: np.ndarray) -> np.ndarray:
    """bf16 / fp16 bit patterns of |x|: the sign bit cleared (exact)."""
    return np.asarray(bits, dtype=np.uint16) & np.uint16(0x7FFF)


def stats(o, lse, o_ref, lse_ref, dtype: str, a_ref=None) -> dict:
    """Error statistics of (o, lse) against the oracle and whether they meet the bar
    (``a_ref``: the oracle's attention of |V|, see ``o_bound``)."""
    o = np.asarray(o, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    d_o = np.abs(o - o_ref)
    bound = o_bound(o_ref, dtype, a_ref)
    excess = d_o - bound if d_o.size else np.zeros(1)
    st = {
        "elements": int(o.size),
        "max_abs_o": float(d_o.max()) if d_o.size else 0.0,
        "max_excess_o": float(excess.max()),
        "relaxed_elements": int((bound > MAX_ABS_O).sum()),
        "rel_l2_o": float(np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-300)),
        "max_abs_lse": float(np.abs(np.asarray(lse, np.float64) - lse_ref).max())
        if np.size(lse) else 0.0,
        "finite": bool(np.isfinite(o).all() and np.isfinite(lse).all()),
    }
    st["ok"] = bool(st["finite"] and st["max_excess_o"] <= 0.0 and st["rel_l2_o"] <= REL_L2_O
                    and st["max_abs_lse"] <= MAX_ABS_LSE)
    return st


# ---------------------------------------------------------------------------------------------
# The backward. No bar is stated for gradients; this one follows from the arithmetic. Each
# gradient passes through a few independent roundings of relative size u: P (or dS) rounded to
# the input type before the product that uses it, and the gradient itself rounded on output.
# Summed over many terms they average out, so the relative L2 error of a gradient stays near
# one u; the bar is 2u, and the largest element error, relative to the largest element of the
# gradient, 6u.
#
# One more term is not of that kind. D_i = <dO_i, O_i> is taken from the forward's stored O,
# whose elements carry the forward's own roundings (at most u A_ic + half a step, <= 2u A_ic
# with A the attention of |V| as above), so |dD_i| <= 2u sum_c |dO_ic| A_ic. dS_ij =
# P_ij (dP_ij - D_i) passes the same dD_i to every key of query i, and dQ_i = scale sum_j dS_ij
# k_j turns it into scale |dD_i| |Kbar_i| with Kbar_i = sum_j P_ij k_j (the attention of K),
# coherent over the keys, while dQ_i itself is a sum that cancels (sum_j P_ij (dP_ij - D_i) =
# 0): for a query that sees few keys, or attends to one key almost alone, this term dominates.
# dQ's error is measured beyond that allowance (``dq_allowance``). In dK_j = scale sum_i dS_ij
# q_i the same errors of the queries that see key j meet with the signs of q and mostly
# average out; where attention is peaked on a few keys and Q is large (the errors of the many
# queries that put almost all their weight on key j then add up against a dK_j that cancels),
# they add about one more u: dK's L2 bar is 3u.
#
# A gradient that vanishes exactly (dQ and dK with a single key, or scale 0) has nothing to
# be relative to: its computed elements must stay below VANISHING_ABS.
GRAD_REL_L2_UNITS = {"dq": 2.0, "dk": 3.0, "dv": 2.0}
GRAD_REL_MAX_UNITS = 6.0
VANISHING_ABS = 1e-3


def grad_bars(dtype: str, grad: str) -> tuple[float, float]:
    """(relative L2 bar, largest-element bar) for gradient ``grad`` ("dq", "dk" or "dv")
    stored in ``dtype``."""
    u = UNIT_ROUNDOFF[dtype]
    return GRAD_REL_L2_UNITS[grad] * u, GRAD_REL_MAX_UNITS * u


def dq_allowance(scale: float, dtype: str, dout, a_ref, kbar) -> np.ndarray:
    """The bound scale * 2u * (sum_c |dO_ic| A_ic) * |Kbar_ic| of dQ's error that comes from D
    through the stored O, for rows i (last axis = features): ``dout`` the upstream gradient's
    values, ``a_ref`` the attention of |V|, ``kbar`` the attention of K, all on those rows."""
    u = UNIT_ROUNDOFF[dtype]
    dout = np.asarray(dout, dtype=np.float64)
    d_err = 2.0 * u * np.sum(np.abs(dout) * np.abs(np.asarray(a_ref, np.float64)), axis=-1,
                             keepdims=True)
    return abs(scale) * d_err * np.abs(np.asarray(kbar, dtype=np.float64))


def grad_stats(g, r, dtype: str, grad: str, allowance=None) -> dict:
    """Error of a computed gradient ``g`` ("dq", "dk" or "dv") against the oracle's ``r`` and
    whether it meets the bars of ``grad_bars``; ``allowance`` (element-wise, e.g.
    ``dq_allowance``) is taken off each element's error first."""
    g = np.asarray(g, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    st = {"finite": bool(np.isfinite(g).all())}
    if np.abs(r).max(initial=0.0) < 1e-6:
        st["vanishing"] = True
        st["max_abs"] = float(np.abs(g).max(initial=0.0))
        st["ok"] = st["finite"] and st["max_abs"] <= VANISHING_ABS
        return st
    l2_bar, max_bar = grad_bars(dtype, grad)
    err = np.abs(g - r)
    st["rel_l2_raw"] = float(np.linalg.norm(err) / np.linalg.norm(r))
    if allowance is not None:
        err = np.maximum(err - np.asarray(allowance, dtype=np.float64), 0.0)
    st["rel_l2"] = float(np.linalg.norm(err) / np.linalg.norm(r))
    st["rel_max"] = float(err.max() / np.abs(r).max())
    st["ok"] = bool(st["finite"] and st["rel_l2"] <= l2_bar and st["rel_max"] <= max_bar)
    return st


# ---------------------------------------------------------------------------------------------
# The oracle's side inputs of the bars above.
def attention_aux(qb, kb, vb, causal, scale, dtype, rows=None, window=(-1, -1),
                  seqlens_k=None):
    """The oracle's attention of |V| (A) and of K (Kbar) on the same Q and K: on every row
    ([B, N, H, d] each) or on the given (b, h, i) rows ([R, d] each)."""
    import oracle
    vabs = magnitude_bits(vb)
    kw = dict(dtype=dtype, window=window, seqlens_k=seqlens_k)
    if rows is None:
        a, _ = oracle.attention(qb, kb, vabs, causal, scale, **kw)
        kbar, _ = oracle.attention(qb, kb, kb, causal, scale, **kw)
    else:
        a, _ = oracle.attention_rows(qb, kb, vabs, rows, causal, scale, **kw)
        kbar, _ = oracle.attention_rows(qb, kb, kb, rows, causal, scale, **kw)
    return a, kbar


def dq_allowance_for(qb, kb, vb, dob, causal, scale, dtype, rows=None, window=(-1, -1),
                     seqlens_k=None):
    """``dq_allowance`` for the inputs' bit patterns (upstream gradient ``dob``), on every row
    ([B, N, H, d]) or on the given (b, h, i) rows ([R, d])."""
    import oracle
    a, kbar = attention_aux(qb, kb, vb, causal, scale, dtype, rows, window, seqlens_k)
    dout = oracle.decode(dob, dtype)
    if rows is not None:
        rows = np.asarray(rows)
        dout = dout[rows[:, 0], rows[:, 2], rows[:, 1]]
    return dq_allowance(scale, dtype, dout, a, kbar)
