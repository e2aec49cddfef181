"""Plant plausible mistakes in a copy of the oracle's C source and check that the pins catch
every one of them (CPU only). The real source is never modified."""
import os

import pytest

import oracle
from pins import ALL_PINS

# (name, exact snippet of attn_oracle.c, replacement)
MUTANTS = [
    ("dropped_max_shift", "l += exp(s[j] - m);", "l += exp(s[j]);"),
    ("normalise_without_shift", "s[j] = exp(s[j] - m) / l;", "s[j] = exp(s[j]) / l;"),
    ("wrong_sign_in_exp", "s[j] = exp(s[j] - m) / l;", "s[j] = exp(m - s[j]) / l;"),
    ("transposed_q_k",
     "for (int64_t c = 0; c < d; ++c) dot += q[q_off + c] * k[k_off + c];",
     "for (int64_t c = 0; c < d; ++c) dot += k[q_off + c] * q[k_off + c];"),
    ("query_row_for_value", "const int64_t v_off = ((b * Nk + j) * H + h) * d;",
     "const int64_t v_off = ((b * Nk + i) * H + h) * d;"),
    ("causal_excludes_diagonal", "if (causal && pos + 1 < z) z = pos + 1;",
     "if (causal && pos < z) z = pos;"),
    ("causal_off_by_one_extra", "if (causal && pos + 1 < z) z = pos + 1;",
     "if (causal && pos + 2 < z) z = pos + 2;"),
    ("window_left_off_by_one", "if (wl >= 0 && pos - wl > a) a = pos - wl;",
     "if (wl >= 0 && pos - wl + 1 > a) a = pos - wl + 1;"),
    ("window_right_ignored", "if (wr >= 0 && pos + wr + 1 < z) z = pos + wr + 1;", ""),
    ("query_position_not_offset",
     "key_range(i + Nk - Nq, causal, window_left, window_right,\n"
     "                          batch_key_length(seqlens_k, b, Nk), &lo, &hi);\n"
     "                attention_row(x.q, x.k, x.v, Nq, Nk, H, d, lo, hi, scale, b, h, i, s,\n"
     "                              o + ((b",
     "key_range(i, causal, window_left, window_right,\n"
     "                          batch_key_length(seqlens_k, b, Nk), &lo, &hi);\n"
     "                attention_row(x.q, x.k, x.v, Nq, Nk, H, d, lo, hi, scale, b, h, i, s,\n"
     "                              o + ((b"),
    ("padding_ignored", "if (!seqlens_k) return N;", "return N;"),
    ("empty_row_lse_zero", "*lse_out = -INFINITY;", "*lse_out = 0.0;"),
    ("scale_dropped", "s[j] = scale * dot;", "s[j] = dot;"),
    ("scale_squared", "s[j] = scale * dot;", "s[j] = scale * scale * dot;"),
    ("lse_without_max", "*lse_out = m + log(l);", "*lse_out = log(l);"),
    ("lse_base2", "*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    ("no_normalisation", "s[j] = exp(s[j] - m) / l;", "s[j] = exp(s[j] - m);"),
    ("head_index_ignored", "const int64_t k_off = ((b * Nk + j) * H + h) * d;",
     "const int64_t k_off = ((b * Nk + j) * H + 0) * d;"),
    ("batch_index_ignored", "const int64_t q_off = ((b * Nq + i) * H + h) * d;",
     "const int64_t q_off = ((0 * Nq + i) * H + h) * d;"),
    ("max_over_prefix_only", "for (int64_t j = lo; j < hi; ++j)\n        if (s[j] > m)",
     "for (int64_t j = lo; j < lo + (hi - lo) / 2; ++j)\n        if (s[j] > m)"),
    ("fp16_bias_wrong", "ldexp((double)(1024 + mant), expo - 25)",
     "ldexp((double)(1024 + mant), expo - 24)"),
    ("fp16_subnormal_wrong", "ldexp((double)mant, -24)", "ldexp((double)mant, -25)"),
    ("bf16_shift_wrong", "(uint32_t)bits << 16", "(uint32_t)bits << 15"),
    ("lse_stride_wrong", "lse + (b * H + h) * Nq + i", "lse + (b * H + h) * Nq + 0"),
    ("bwd_drops_D", "dS[i * N + j] = P[i * N + j] * (dS[i * N + j] - Di);",
     "dS[i * N + j] = P[i * N + j] * dS[i * N + j];"),
    ("bwd_dq_unscaled", "for (int64_t c = 0; c < d; ++c) out[c] *= scale;", ""),
    ("bwd_dv_from_dS", "const double ds = dS[i * N + j], p = P[i * N + j];",
     "const double ds = dS[i * N + j], p = dS[i * N + j];"),
    ("bwd_dk_transposed", "const double ds = dS[i * N + j], p = P[i * N + j];",
     "const double ds = dS[j * N + i], p = P[i * N + j];"),
    ("bwd_sampled_drops_D", "const double ds = p * (dp - D[i]);", "const double ds = p * dp;"),
    ("bwd_sampled_key_left_bound_ignored", "if (j < lo || j >= hi) continue;",
     "if (j >= hi) continue;"),
    ("bwd_sampled_key_right_bound_off_by_one", "if (j < lo || j >= hi) continue;",
     "if (j < lo || j > hi) continue;"),
]


def test_real_source_passes_every_pin(oracle_lib):
    pytest.importorskip("mpmath")
    for pin in ALL_PINS:
        pin(oracle_lib)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    pytest.importorskip("mpmath")
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, "mutation site must be unique: %r" % old
    mutated = tmp_path / ("oracle_%s.c" % name)
    mutated.write_text(src.replace(old, new))
    lib = oracle.load(oracle.compile_library(str(mutated), str(tmp_path / ("lib_%s.so" % name))))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, "no pin catches the mutant %s" % name
