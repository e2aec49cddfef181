"""Pins for the attention oracle: checks against facts fixed by the pages and by mathematics.

Each pin takes a loaded oracle library (``oracle.load()`` or a mutated build of the same
source) and raises AssertionError when the oracle disagrees with the fact. None of them
retypes the oracle's formula: they use closed forms, invariants, special cases with known
answers, the method's tiled algorithm (a different evaluation order that the pages state
reaches the same result), an independent arbitrary-precision evaluation without the max
shift, and library conversions.

Sources of the facts ("FlashAttention 优化原理与实现要点解析" unless noted):
  §1  Attention(Q,K,V) = Softmax(QK^T/sqrt(d)) V; tiling does not change the result.
  §4.1 softmax definition: rows of P are positive and sum to 1.
  §4.2-§5 online softmax / tiled attention reach the exact softmax.
  §7  causal: query i attends to keys j <= i.
  "FlashAttention V2 核心原理与架构设计" §2.1: the element-wise online softmax.
  "FlashAttention V2 核心原理与架构设计" §2.3: per-row statistics m and l are kept
      (reported as LSE = m + ln l).
"""
from __future__ import annotations

import math

import numpy as np

import oracle


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _attn(lib, q, k, v, causal, scale):
    return oracle.attention(q, k, v, causal, scale, lib=lib)


# ---------------------------------------------------------------------------------------------
def pin_decode_fp16(lib):
    """fp16 decoding equals numpy's float16 -> float64 conversion for every bit pattern."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, "fp16", lib=lib)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_decode_bf16(lib):
    """bf16 decoding equals torch's bfloat16 -> float64 conversion for every bit pattern."""
    import torch
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, "bf16", lib=lib)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_probability_rows(lib):
    """With V = I (d = N), O[i, :] is row i of P: non-negative, summing to 1; causal rows
    put exactly zero weight on keys j > i."""
    N = 24
    rng = _rng(11)
    q = rng.standard_normal((2, N, 2, N))
    k = rng.standard_normal((2, N, 2, N))
    v = np.broadcast_to(np.eye(N)[None, :, None, :], (2, N, 2, N)).copy()
    for causal in (False, True):
        P, _ = _attn(lib, q, k, v, causal, 0.3)
        assert (P >= 0).all()
        assert np.abs(P.sum(axis=-1) - 1.0).max() < 1e-14
        if causal:
            upper = np.triu(np.ones((N, N), dtype=bool), 1)
            assert (P.transpose(0, 2, 1, 3)[:, :, upper] == 0).all()
        else:
            assert (P > 0).all()


def pin_zero_queries(lib):
    """Q = 0 makes every score 0: O is the mean of the allowed V rows, LSE = ln(#keys)."""
    B, N, H, d = 2, 37, 3, 8
    rng = _rng(12)
    q = np.zeros((B, N, H, d))
    k = rng.standard_normal((B, N, H, d))
    v = rng.standard_normal((B, N, H, d))
    o, lse = _attn(lib, q, k, v, False, 0.125)
    assert np.abs(o - v.mean(axis=1, keepdims=True)).max() < 1e-13
    assert np.abs(lse - math.log(N)).max() < 1e-13
    o, lse = _attn(lib, q, k, v, True, 0.125)
    prefix_mean = np.cumsum(v, axis=1) / np.arange(1, N + 1)[None, :, None, None]
    assert np.abs(o - prefix_mean).max() < 1e-13
    assert np.abs(lse - np.log(np.arange(1, N + 1))[None, None, :]).max() < 1e-13


def pin_constant_values(lib):
    """V rows all equal to one vector c: O = c for every row, causal or not."""
    B, N, H, d = 1, 29, 2, 16
    rng = _rng(13)
    q = 3 * rng.standard_normal((B, N, H, d))
    k = rng.standard_normal((B, N, H, d))
    c = rng.standard_normal((1, 1, H, d))
    v = np.broadcast_to(c, (B, N, H, d)).copy()
    for causal in (False, True):
        o, _ = _attn(lib, q, k, v, causal, 0.25)
        assert np.abs(o - c).max() < 1e-13


def pin_causal_first_row(lib):
    """Causal row 0 sees only key 0: O[0] = V[0] and LSE[0] = scale * <q_0, k_0>."""
    B, N, H, d = 2, 17, 2, 8
    rng = _rng(14)
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    scale = 0.35
    o, lse = _attn(lib, q, k, v, True, scale)
    assert np.abs(o[:, 0] - v[:, 0]).max() < 1e-15
    want = scale * np.einsum("bhc,bhc->bh", q[:, 0], k[:, 0])
    assert np.abs(lse[:, :, 0] - want).max() < 1e-13


def pin_single_token(lib):
    """N = 1: O = V and LSE = scale * <q, k>, causal or not."""
    rng = _rng(15)
    q, k, v = (rng.standard_normal((3, 1, 2, 5)) for _ in range(3))
    for causal in (False, True):
        o, lse = _attn(lib, q, k, v, causal, 0.7)
        assert np.abs(o - v).max() < 1e-15
        want = 0.7 * np.einsum("bnhc,bnhc->bhn", q, k)
        assert np.abs(lse - want).max() < 1e-13


def pin_two_key_closed_form(lib):
    """One query, two keys with scores 0 and 1: p = (1, e) / (1 + e), so
    O = (v0 + e v1) / (1 + e) and LSE = ln(1 + e)."""
    q = np.array([[[[1.0]]], [[[1.0]]]]).reshape(1, 2, 1, 1)
    k = np.array([0.0, 1.0]).reshape(1, 2, 1, 1)
    v = np.array([2.0, -3.0]).reshape(1, 2, 1, 1)
    o, lse = _attn(lib, q, k, v, False, 1.0)
    e = math.e
    assert abs(o[0, 0, 0, 0] - (2.0 - 3.0 * e) / (1 + e)) < 1e-15
    assert abs(lse[0, 0, 0] - math.log(1 + e)) < 1e-15
    # causal: row 0 sees only key 0 (score 0): O = v0, LSE = 0
    o, lse = _attn(lib, q, k, v, True, 1.0)
    assert o[0, 0, 0, 0] == 2.0 and lse[0, 0, 0] == 0.0
    assert abs(o[0, 1, 0, 0] - (2.0 - 3.0 * e) / (1 + e)) < 1e-15


def pin_key_shift(lib):
    """Adding one vector w to every key row adds scale*<q_i, w> to row i's scores: O is
    unchanged and LSE_i grows by exactly that amount (softmax is shift invariant)."""
    B, N, H, d = 1, 40, 2, 8
    rng = _rng(16)
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    w = rng.standard_normal((1, 1, H, d))
    scale = 0.5
    for causal in (False, True):
        o0, l0 = _attn(lib, q, k, v, causal, scale)
        o1, l1 = _attn(lib, q, k + w, v, causal, scale)
        assert np.abs(o1 - o0).max() < 1e-12
        shift = scale * np.einsum("bnhc,bnhc->bhn", q, np.broadcast_to(w, q.shape))
        assert np.abs((l1 - l0) - shift).max() < 1e-12


def pin_kv_permutation(lib):
    """Non-causal attention is invariant under one permutation applied to the rows of K
    and V together."""
    B, N, H, d = 2, 33, 2, 8
    rng = _rng(17)
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    perm = rng.permutation(N)
    o0, l0 = _attn(lib, q, k, v, False, 0.4)
    o1, l1 = _attn(lib, q, k[:, perm], v[:, perm], False, 0.4)
    assert np.abs(o1 - o0).max() < 1e-13
    assert np.abs(l1 - l0).max() < 1e-13


def _brute_force_mp(q, k, v, causal, scale, allowed=None):
    """sum_j e^{s_j} v_j / sum_j e^{s_j} in 60-digit arithmetic, no max shift. ``allowed``
    (b, i, j) -> bool restricts the keys (default: all, or j <= i when causal); a row with no
    allowed key gives O = 0, LSE = -inf."""
    import mpmath
    mp = mpmath.mp.clone()
    mp.dps = 60
    B, N, H, d = q.shape
    o = np.zeros((B, N, H, d))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                if allowed is None:
                    js = list(range(i + 1) if causal else range(N))
                else:
                    js = [j for j in range(N) if allowed(b, i, j)]
                if not js:
                    lse[b, h, i] = -math.inf
                    continue
                ws = []
                for j in js:
                    s = mp.mpf(0)
                    for c in range(d):
                        s += mp.mpf(float(q[b, i, h, c])) * mp.mpf(float(k[b, j, h, c]))
                    ws.append(mp.exp(mp.mpf(scale) * s))
                den = mp.fsum(ws)
                for c in range(d):
                    num = mp.fsum(wj * mp.mpf(float(v[b, j, h, c])) for wj, j in zip(ws, js))
                    o[b, i, h, c] = float(num / den)
                lse[b, h, i] = float(mp.log(den))
    return o, lse


def pin_brute_force_small(lib):
    """N <= 16, several heads and batches: equals an independent 60-digit evaluation of the
    definition without the max shift, both masks, moderate logits."""
    rng = _rng(18)
    for (B, N, H, d) in [(1, 1, 1, 4), (2, 7, 3, 5), (1, 16, 2, 8)]:
        q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
        for causal in (False, True):
            o, lse = _attn(lib, q, k, v, causal, 0.6)
            ob, lb = _brute_force_mp(q, k, v, causal, 0.6)
            assert np.abs(o - ob).max() < 1e-12
            assert np.abs(lse - lb).max() < 1e-12


def pin_brute_force_large_logits(lib):
    """Scores in the thousands (e^s overflows float64 without the max shift): the oracle
    stays finite and matches the 60-digit evaluation, which needs no shift."""
    rng = _rng(19)
    B, N, H, d = 1, 12, 2, 4
    q = 40 * rng.standard_normal((B, N, H, d))
    k = 40 * rng.standard_normal((B, N, H, d))
    v = rng.standard_normal((B, N, H, d))
    for causal in (False, True):
        o, lse = _attn(lib, q, k, v, causal, 0.5)
        ob, lb = _brute_force_mp(q, k, v, causal, 0.5)
        assert np.isfinite(o).all() and np.isfinite(lse).all()
        assert np.abs(o - ob).max() < 1e-12
        assert (np.abs(lse - lb) / np.maximum(1.0, np.abs(lb))).max() < 1e-13


def pin_tiled_algorithm(lib):
    """The pages' tiled online-softmax algorithm (Q blocks outer, K/V blocks inner, causal
    block skip, normalisation at the end) reaches the plain definition: several block shapes,
    ragged tails, both masks."""
    rng = _rng(20)
    N, d = 45, 8
    q, k, v = (rng.standard_normal((1, N, 1, d)) for _ in range(3))
    for causal in (False, True):
        o, lse = _attn(lib, q, k, v, causal, 0.4)
        for Br, Bc in [(1, 1), (8, 8), (16, 7), (45, 45), (64, 16)]:
            ot, lt = oracle.blockwise_attention(q[0, :, 0], k[0, :, 0], v[0, :, 0], Br, Bc,
                                                causal, 0.4)
            assert np.abs(ot - o[0, :, 0]).max() < 1e-12
            assert np.abs(lt - lse[0, 0]).max() < 1e-12


def pin_torch_math_sdpa(lib):
    """Third opinion: torch's math scaled_dot_product_attention in float64 on the CPU."""
    import torch
    rng = _rng(21)
    B, N, H, d = 2, 50, 3, 16
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    for causal in (False, True):
        o, _ = _attn(lib, q, k, v, causal, 0.3)
        t = [torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v)]
        ref = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=causal, scale=0.3)
        assert np.abs(o - ref.permute(0, 2, 1, 3).numpy()).max() < 1e-12


def pin_dtype_inputs(lib):
    """Bit-pattern inputs give the same result as their exactly decoded values, for both
    storage types, and the selected-rows entry point matches the full one."""
    from io_aware_attention_fa2_gb300.inputs import make_qkv
    for dtype in ("bf16", "fp16"):
        qb, kb, vb = make_qkv(1, 2, 20, 8, dtype, seed=7, q_scale=2.0)
        o_bits, l_bits = oracle.attention(qb, kb, vb, True, 0.3, dtype=dtype, lib=lib)
        dec = [oracle.decode(x, dtype, lib=lib) for x in (qb, kb, vb)]
        o_f, l_f = _attn(lib, *dec, True, 0.3)
        assert np.array_equal(o_bits, o_f) and np.array_equal(l_bits, l_f)
        rows = np.array([[0, 1, 19], [0, 0, 0], [0, 1, 7]])
        o_r, l_r = oracle.attention_rows(qb, kb, vb, rows, True, 0.3, dtype=dtype, lib=lib)
        for t, (b, h, i) in enumerate(rows):
            assert np.array_equal(o_r[t], o_bits[b, i, h]) and l_r[t] == l_bits[b, h, i]


def pin_padding_is_truncation(lib):
    """Per-batch key lengths (padding mask) give, for every query, exactly the attention over
    the first len_b keys and values; a zero length gives O = 0, LSE = -inf."""
    B, N, H, d = 3, 21, 2, 8
    rng = _rng(22)
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    lens = [21, 9, 0]
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal, 0.4, lib=lib, seqlens_k=lens)
        for b, L in enumerate(lens):
            if L == 0:
                assert (o[b] == 0).all() and (lse[b] == -np.inf).all()
                continue
            # queries keep all N positions; keys and values are cut to the first L rows
            for i in range(N):
                ob, lb = _brute_force_rows(q[b], k[b, :L], v[b, :L], causal, 0.4, i)
                assert np.abs(o[b, i] - ob).max() < 1e-12
                assert np.abs(lse[b, :, i] - lb).max() < 1e-12


def _brute_force_rows(qb, kb, vb, causal, scale, i):
    """Row i of attention for one batch (all heads) in float64, keys [0, len(kb)), direct
    softmax via numpy (no shared code with the oracle)."""
    L, H = kb.shape[0], qb.shape[1]
    o = np.zeros((H, qb.shape[2]))
    lse = np.full(H, -np.inf)
    js = [j for j in range(L) if (not causal or j <= i)]
    if not js:
        return o, lse
    for h in range(H):
        sc = np.array([scale * float(qb[i, h] @ kb[j, h]) for j in js])
        mx = sc.max()
        w = np.exp(sc - mx)
        o[h] = (w[:, None] * vb[js, h]).sum(0) / w.sum()
        lse[h] = mx + math.log(w.sum())
    return o, lse


def pin_sliding_window_brute_force(lib):
    """Sliding windows (left / right bounds, with and without causal) equal the 60-digit
    brute force over the explicitly listed allowed keys, including rows left empty."""
    rng = _rng(23)
    B, N, H, d = 1, 14, 2, 6
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    lens = [11]
    for causal, (left, right) in [(True, (3, -1)), (False, (2, 4)), (False, (-1, 1)),
                                  (True, (0, -1)), (False, (5, 0)), (True, (2, 1))]:
        def allowed(b, i, j, causal=causal, left=left, right=right):
            return (j < lens[b] and (not causal or j <= i) and (left < 0 or j >= i - left)
                    and (right < 0 or j <= i + right))
        o, lse = oracle.attention(q, k, v, causal, 0.5, lib=lib, window=(left, right),
                                  seqlens_k=lens)
        ob, lb = _brute_force_mp(q, k, v, causal, 0.5, allowed=allowed)
        assert np.abs(o - ob).max() < 1e-12
        fin = np.isfinite(lb)
        assert np.array_equal(fin, np.isfinite(lse))
        assert np.abs(lse[fin] - lb[fin]).max() < 1e-12


def pin_window_special_cases(lib):
    """Causal with window_left = 0: each query sees only itself (O = V_i, LSE = scale <q_i,
    k_i>); windows at least N wide change nothing."""
    rng = _rng(24)
    B, N, H, d = 2, 19, 2, 8
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, True, 0.3, lib=lib, window=(0, -1))
    assert np.abs(o - v).max() < 1e-15
    assert np.abs(lse - 0.3 * np.einsum("bnhc,bnhc->bhn", q, k)).max() < 1e-13
    for causal in (False, True):
        o0, l0 = oracle.attention(q, k, v, causal, 0.3, lib=lib)
        o1, l1 = oracle.attention(q, k, v, causal, 0.3, lib=lib, window=(N, N))
        assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def pin_tiled_algorithm_masks(lib):
    """The tiled algorithm with padding / window masks and block skipping reaches the plain
    definition, for ragged block shapes."""
    rng = _rng(25)
    N, d = 41, 8
    q, k, v = (rng.standard_normal((1, N, 1, d)) for _ in range(3))
    for causal, window, L in [(True, (7, -1), 41), (False, (5, 5), 30), (True, (-1, -1), 17),
                              (False, (-1, 0), 41), (True, (3, -1), 2)]:
        o, lse = oracle.attention(q, k, v, causal, 0.4, lib=lib, window=window, seqlens_k=[L])
        for Br, Bc in [(8, 8), (16, 7), (64, 16)]:
            ot, lt = oracle.blockwise_attention(q[0, :, 0], k[0, :, 0], v[0, :, 0], Br, Bc,
                                                causal, 0.4, window=window, kv_len=L)
            assert np.abs(ot - o[0, :, 0]).max() < 1e-12
            fin = np.isfinite(lse[0, 0])
            assert np.array_equal(fin, np.isfinite(lt))
            assert np.abs(lt[fin] - lse[0, 0][fin]).max() < 1e-12


ALL_PINS = [
    pin_decode_fp16, pin_decode_bf16, pin_probability_rows, pin_zero_queries,
    pin_constant_values, pin_causal_first_row, pin_single_token, pin_two_key_closed_form,
    pin_key_shift, pin_kv_permutation, pin_brute_force_small, pin_brute_force_large_logits,
    pin_tiled_algorithm, pin_torch_math_sdpa, pin_dtype_inputs, pin_padding_is_truncation,
    pin_sliding_window_brute_force, pin_window_special_cases, pin_tiled_algorithm_masks,
]


def pin_fewer_queries_brute_force(lib):
    """Nq < Nk (queries are the last Nq positions): equals the 60-digit brute force over the
    allowed keys of position i + Nk - Nq, for causal, window and padding."""
    rng = _rng(26)
    B, Nq, Nk, H, d = 2, 3, 13, 2, 6
    q = rng.standard_normal((B, Nq, H, d))
    k, v = (rng.standard_normal((B, Nk, H, d)) for _ in range(2))
    lens = [13, 9]
    for causal, (left, right) in [(True, (-1, -1)), (False, (-1, -1)), (True, (4, -1)),
                                  (False, (2, 1))]:
        def allowed(b, i, j, causal=causal, left=left, right=right):
            p = i + Nk - Nq
            return (j < lens[b] and (not causal or j <= p) and (left < 0 or j >= p - left)
                    and (right < 0 or j <= p + right))
        o, lse = oracle.attention(q, k, v, causal, 0.5, lib=lib, window=(left, right),
                                  seqlens_k=lens)
        ob, lb = _brute_force_mp_qk(q, k, v, 0.5, allowed)
        assert np.abs(o - ob).max() < 1e-12
        fin = np.isfinite(lb)
        assert np.array_equal(fin, np.isfinite(lse))
        assert np.abs(lse[fin] - lb[fin]).max() < 1e-12


def _brute_force_mp_qk(q, k, v, scale, allowed):
    import mpmath
    mp = mpmath.mp.clone()
    mp.dps = 60
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    o = np.zeros((B, Nq, H, d))
    lse = np.full((B, H, Nq), -math.inf)
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                js = [j for j in range(Nk) if allowed(b, i, j)]
                if not js:
                    continue
                ws = [mp.exp(mp.mpf(scale) * mp.fsum(mp.mpf(float(q[b, i, h, c])) *
                                                     mp.mpf(float(k[b, j, h, c]))
                                                     for c in range(d))) for j in js]
                den = mp.fsum(ws)
                for c in range(d):
                    o[b, i, h, c] = float(mp.fsum(w * mp.mpf(float(v[b, j, h, c]))
                                                  for w, j in zip(ws, js)) / den)
                lse[b, h, i] = float(mp.log(den))
    return o, lse


def pin_fewer_queries_are_last_rows(lib):
    """Attention of the last Nq queries against all Nk keys equals the last Nq rows of the
    square (Nq = Nk) attention whose final queries are those Nq, for every mask."""
    rng = _rng(27)
    B, Nk, H, d = 2, 37, 2, 8
    q_full, k, v = (rng.standard_normal((B, Nk, H, d)) for _ in range(3))
    for Nq in (1, 5, 37):
        q = q_full[:, Nk - Nq:]
        for causal, window, lens in [(True, (-1, -1), None), (False, (6, 3), [37, 20]),
                                     (True, (10, -1), [30, 37])]:
            o, lse = oracle.attention(q, k, v, causal, 0.3, lib=lib, window=window,
                                      seqlens_k=lens)
            of, lf = oracle.attention(q_full, k, v, causal, 0.3, lib=lib, window=window,
                                      seqlens_k=lens)
            assert np.array_equal(o, of[:, Nk - Nq:]) and np.array_equal(lse, lf[:, :, Nk - Nq:])


def pin_tiled_algorithm_fewer_queries(lib):
    """The tiled algorithm with Nq < Nk (query blocks at the end of the key sequence)
    reaches the plain definition."""
    rng = _rng(28)
    Nq, Nk, d = 11, 40, 8
    q = rng.standard_normal((1, Nq, 1, d))
    k, v = (rng.standard_normal((1, Nk, 1, d)) for _ in range(2))
    for causal, window in [(True, (-1, -1)), (False, (9, 2)), (True, (5, -1))]:
        o, lse = oracle.attention(q, k, v, causal, 0.4, lib=lib, window=window)
        for Br, Bc in [(4, 8), (16, 7)]:
            ot, lt = oracle.blockwise_attention(q[0, :, 0], k[0, :, 0], v[0, :, 0], Br, Bc,
                                                causal, 0.4, window=window)
            assert np.abs(ot - o[0, :, 0]).max() < 1e-12
            assert np.abs(lt - lse[0, 0]).max() < 1e-12


ALL_PINS += [pin_fewer_queries_brute_force, pin_fewer_queries_are_last_rows,
             pin_tiled_algorithm_fewer_queries]


# --------------------------------------------------------------------------------- backward
def _loss(lib, q, k, v, dout, causal, scale, window=(-1, -1), lens=None):
    o, _ = oracle.attention(q, k, v, causal, scale, lib=lib, window=window, seqlens_k=lens)
    return float((o * dout).sum())


def pin_bwd_finite_differences(lib):
    """dQ, dK, dV equal central differences of L = sum(dO * O) computed with the forward
    (which is pinned on its own), on random elements, for several masks."""
    rng = _rng(30)
    B, N, H, d = 2, 9, 2, 5
    q, k, v, dout = (rng.standard_normal((B, N, H, d)) for _ in range(4))
    for causal, window, lens in [(False, (-1, -1), None), (True, (-1, -1), None),
                                 (True, (3, -1), [9, 6])]:
        dq, dk, dv = oracle.attention_bwd(q, k, v, dout, causal, 0.45, lib=lib, window=window,
                                          seqlens_k=lens)
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for _ in range(12):
                idx = tuple(int(rng.integers(0, n)) for n in x.shape)
                h = 1e-5
                x0 = x[idx]
                x[idx] = x0 + h
                lp = _loss(lib, q, k, v, dout, causal, 0.45, window, lens)
                x[idx] = x0 - h
                lm = _loss(lib, q, k, v, dout, causal, 0.45, window, lens)
                x[idx] = x0
                fd = (lp - lm) / (2 * h)
                assert abs(fd - g[idx]) <= 1e-7 * max(1.0, abs(fd)), (name, causal, idx, fd, g[idx])


def pin_bwd_identities(lib):
    """Rows of P sum to 1, so sum over keys of dV = sum over queries of dO and sum over keys of
    dK = 0 (softmax ignores a common shift); with all keys equal P does not depend on Q, so
    dQ = 0; with N = 1, dV = dO and dQ = dK = 0."""
    rng = _rng(31)
    B, N, H, d = 2, 23, 3, 8
    q, k, v, dout = (rng.standard_normal((B, N, H, d)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = oracle.attention_bwd(q, k, v, dout, causal, 0.3, lib=lib)
        assert np.abs(dv.sum(axis=1) - dout.sum(axis=1)).max() < 1e-12
        assert np.abs(dk.sum(axis=1)).max() < 1e-12
        k_eq = np.broadcast_to(k[:, :1], k.shape).copy()
        dq0, _, _ = oracle.attention_bwd(q, k_eq, v, dout, causal, 0.3, lib=lib)
        assert np.abs(dq0).max() < 1e-13
    q1, k1, v1, do1 = (x[:, :1] for x in (q, k, v, dout))
    dq, dk, dv = oracle.attention_bwd(q1, k1, v1, do1, True, 0.3, lib=lib)
    assert np.array_equal(dv, do1) and not dq.any() and not dk.any()


def pin_bwd_matches_torch_autograd(lib):
    """Third opinion: torch autograd through math attention in float64 on the CPU."""
    import torch
    rng = _rng(32)
    B, N, H, d = 2, 17, 2, 8
    q, k, v, dout = (rng.standard_normal((B, N, H, d)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = oracle.attention_bwd(q, k, v, dout, causal, 0.35, lib=lib)
        t = [torch.from_numpy(x.copy()).permute(0, 2, 1, 3).requires_grad_() for x in (q, k, v)]
        o = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=causal, scale=0.35)
        o.backward(torch.from_numpy(dout).permute(0, 2, 1, 3))
        for g, ref in zip((dq, dk, dv), t):
            assert np.abs(g - ref.grad.permute(0, 2, 1, 3).numpy()).max() < 1e-12


def pin_bwd_sampled_matches_full(lib):
    """The sampled backward (no N x N storage, used at full sizes) equals the full backward's
    gradients at the sampled positions, causal or not, with and without a window and key
    lengths (one batch with no key at all), on real and on bf16 inputs."""
    from io_aware_attention_fa2_gb300.inputs import round_to_bits
    rng = _rng(33)
    B, N, H, d = 2, 41, 3, 8
    real = [rng.standard_normal((B, N, H, d)) for _ in range(4)]
    heads, keys, queries = [(0, 0), (1, 2), (0, 1)], [0, 1, 20, 29, 39, 40], [0, 2, 21, 40]
    masks = [((-1, -1), None), ((5, 3), None), ((-1, -1), [30, 41]), ((6, 0), [41, 0])]
    for dtype in (None, "bf16"):
        args = real if dtype is None else [round_to_bits(x, "bf16") for x in real]
        for causal in (False, True):
            for window, lens in masks:
                dq, dk, dv = oracle.attention_bwd(*args, causal, 0.37, dtype=dtype, lib=lib,
                                                  window=window, seqlens_k=lens)
                sq, sk, sv = oracle.attention_bwd_sampled(
                    *args, causal, 0.37, heads, keys, queries, dtype=dtype, lib=lib,
                    window=window, seqlens_k=lens)
                for t, (b, h) in enumerate(heads):
                    assert np.abs(sq[t] - dq[b, queries, h]).max() < 1e-12
                    assert np.abs(sk[t] - dk[b, keys, h]).max() < 1e-12
                    assert np.abs(sv[t] - dv[b, keys, h]).max() < 1e-12


ALL_PINS += [pin_bwd_finite_differences, pin_bwd_identities, pin_bwd_matches_torch_autograd,
             pin_bwd_sampled_matches_full]
