/*
 * attn_oracle.c -- plain fp64 CPU attention: the oracle for the fused attention forward.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg load this file's library. The product path (the CUDA library) never calls it, and the
 * two share no code, header, table or constant.
 *
 * What it computes is the plain definition of scaled dot-product attention, evaluated in
 * double precision on the exact values of the bf16/fp16 inputs:
 *
 *   "FlashAttention 优化原理与实现要点解析" §1: Attention(Q,K,V) = Softmax(Q K^T / sqrt(d)) V,
 *       here with the caller's scale in place of 1/sqrt(d).
 *   same page §2: three steps, S = Q K^T, P = Softmax(S), O = P V, materialising S and P
 *       (one row of each at a time: row i of O depends only on row i of S and P).
 *   same page §4.1: Softmax(x_i) = e^{x_i} / sum_j e^{x_j}, evaluated as the three passes it
 *       lists: (1) the row maximum m, (2) the sum l = sum_j e^{x_j - m}, (3) e^{x_i - m} / l.
 *   same page §7: causal masking, a query attends only to keys at positions <= its own.
 *   "FlashAttention V2 核心原理与架构设计" §2.3: the kernel also keeps the per-row softmax
 *       denominator l and row maximum m; the oracle reports them as one log-sum-exp,
 *       LSE_i = m_i + ln(l_i), in units of scaled scores.
 *   "FlashAttention 优化原理与实现要点解析" §8 names the mask kinds an implementation may
 *       support: causal,
 *       padding and sliding-window masks. The oracle takes all three as one rule per query:
 *       key j is allowed for query i of batch b when j < len_b (padding: keys at or past the
 *       batch's key length do not exist; len_b = N without a length array), j <= i (causal),
 *       j >= i - window_left (window_left >= 0) and j <= i + window_right (window_right >= 0).
 *       The allowed keys always form one interval [lo, hi). A row with no allowed key has
 *       O = 0 and LSE = -inf (the sum l is 0).
 *   "FlashAttention V2 核心原理与架构设计" §5.1 (combining with FlashDecoding for long
 *       sequences): queries may be fewer than keys (Nq <= Nk, e.g. decoding). The queries are
 *       then the last Nq positions of the sequence: query i sits at position i + Nk - Nq, and
 *       the causal and window bounds above are taken relative to that position.
 *
 * Layouts: q and o are [B, Nq, H, d], k and v [B, Nk, H, d], row-major (element (b, n, h, c)
 * at ((b*N + n)*H + h)*d + c with N the tensor's own length); lse is [B, H, Nq]; the optional
 * key lengths are int32 [B].
 *
 * There is no blocking, fusion or reordering here: one (b, h, i) row at a time, the three
 * passes in order. Rows are independent, so OpenMP spreads rows over host cores. The bf16 /
 * fp16 inputs are decoded to their exact fp64 values once per call, before any arithmetic
 * (decoding is exact, so this changes no result, only the cost of re-reading an element).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F64 = 0, ORACLE_BF16 = 1, ORACLE_FP16 = 2 };

/* bfloat16 is the upper half of an IEEE binary32: sign, 8 exponent bits, 7 mantissa bits. */
static double bf16_bits_value(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* IEEE binary16: sign, 5 exponent bits (bias 15), 10 mantissa bits. */
static double fp16_bits_value(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int mant = bits & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)mant, -24);                 /* subnormal: mant * 2^-14 * 2^-10 */
    else if (expo == 31)
        mag = mant ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + mant), expo - 25);  /* (1 + mant/1024) * 2^(expo-15) */
    return sign ? -mag : mag;
}

static double elem(const void* base, int kind, int64_t idx) {
    switch (kind) {
    case ORACLE_BF16: return bf16_bits_value(((const uint16_t*)base)[idx]);
    case ORACLE_FP16: return fp16_bits_value(((const uint16_t*)base)[idx]);
    default: return ((const double*)base)[idx];
    }
}

int oracle_decode(const uint16_t* bits, int64_t n, int kind, double* out) {
    if (!bits || !out || n < 0) return -1;
    if (kind != ORACLE_BF16 && kind != ORACLE_FP16) return -2;
    for (int64_t t = 0; t < n; ++t) out[t] = elem(bits, kind, t);
    return 0;
}

/* The exact fp64 values of n input elements of the given kind. fp64 inputs are used in place
 * (*owned = 0); bf16 / fp16 ones are decoded into a new array (*owned = 1, free it). Returns
 * NULL when memory runs out. */
static const double* as_f64(const void* base, int kind, int64_t n, int* owned) {
    *owned = 0;
    if (kind == ORACLE_F64) return (const double*)base;
    double* out = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!out) return NULL;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) out[t] = elem(base, kind, t);
    *owned = 1;
    return out;
}

/* The decoded inputs of one call. */
typedef struct {
    const double *q, *k, *v, *g;   /* g: the upstream gradient (backward only) */
    int own_q, own_k, own_v, own_g;
} Decoded;

static void release(Decoded* x) {
    if (x->own_q) free((void*)x->q);
    if (x->own_k) free((void*)x->k);
    if (x->own_v) free((void*)x->v);
    if (x->own_g) free((void*)x->g);
}

/* Decode q (nq elements), k, v (nk each) and optionally dout (nq). Returns 0 or -4. */
static int decode_inputs(const void* q, const void* k, const void* v, const void* dout, int kind,
                         int64_t nq, int64_t nk, Decoded* x) {
    memset(x, 0, sizeof *x);
    x->q = as_f64(q, kind, nq, &x->own_q);
    x->k = as_f64(k, kind, nk, &x->own_k);
    x->v = as_f64(v, kind, nk, &x->own_v);
    if (dout) x->g = as_f64(dout, kind, nq, &x->own_g);
    if (!x->q || !x->k || !x->v || (dout && !x->g)) {
        release(x);
        return -4;
    }
    return 0;
}

/* The keys query i may attend to: [lo, hi). `len_b` is the batch's key length; `pos` is the
 * query's position in the key sequence (i + Nk - Nq). */
static void key_range(int64_t pos, int causal, int64_t wl, int64_t wr, int64_t len_b,
                      int64_t* lo, int64_t* hi) {
    int64_t a = 0, z = len_b;
    if (causal && pos + 1 < z) z = pos + 1;
    if (wl >= 0 && pos - wl > a) a = pos - wl;
    if (wr >= 0 && pos + wr + 1 < z) z = pos + wr + 1;
    *lo = a;
    *hi = z;
}

/* One output row: query i of head (b, h) over keys [lo, hi). `s` is scratch of >= Nk doubles. */
static void attention_row(const double* q, const double* k, const double* v,
                          int64_t Nq, int64_t Nk, int64_t H, int64_t d, int64_t lo, int64_t hi,
                          double scale, int64_t b, int64_t h, int64_t i, double* s,
                          double* o_row, double* lse_out) {
    const int64_t q_off = ((b * Nq + i) * H + h) * d;
    if (lo >= hi) {             /* no key allowed: O = 0, LSE = -inf */
        for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
        *lse_out = -INFINITY;
        return;
    }

    /* Step 1: S[i, j] = scale * <q_i, k_j>. */
    for (int64_t j = lo; j < hi; ++j) {
        const int64_t k_off = ((b * Nk + j) * H + h) * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += q[q_off + c] * k[k_off + c];
        s[j] = scale * dot;
    }

    /* Softmax pass 1: the row maximum. */
    double m = -INFINITY;
    for (int64_t j = lo; j < hi; ++j)
        if (s[j] > m) m = s[j];

    /* Softmax pass 2: the sum of exponentials relative to the maximum. */
    double l = 0.0;
    for (int64_t j = lo; j < hi; ++j) l += exp(s[j] - m);

    /* Softmax pass 3: normalise, turning S[i, :] into P[i, :] in place. */
    for (int64_t j = lo; j < hi; ++j) s[j] = exp(s[j] - m) / l;

    /* Step 3: O[i, :] = P[i, :] V. */
    for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
    for (int64_t j = lo; j < hi; ++j) {
        const int64_t v_off = ((b * Nk + j) * H + h) * d;
        for (int64_t c = 0; c < d; ++c) o_row[c] += s[j] * v[v_off + c];
    }

    *lse_out = m + log(l);
}

static int64_t batch_key_length(const int32_t* seqlens_k, int64_t b, int64_t N) {
    if (!seqlens_k) return N;
    int64_t len = seqlens_k[b];
    return len < 0 ? 0 : (len > N ? N : len);
}

static int check_args(const void* q, const void* k, const void* v, int kind, int64_t B,
                      int64_t H, int64_t Nq, int64_t Nk, int64_t d) {
    if (!q || !k || !v) return -1;
    if (kind != ORACLE_F64 && kind != ORACLE_BF16 && kind != ORACLE_FP16) return -2;
    if (B < 1 || H < 1 || Nq < 1 || Nk < Nq || d < 1) return -3;
    return 0;
}

/* Full attention, Nq queries against Nk >= Nq keys, general mask: o [B, Nq, H, d],
 * lse [B, H, Nq]. */
int oracle_attention_qk(const void* q, const void* k, const void* v, int kind, int64_t B,
                        int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal,
                        int64_t window_left, int64_t window_right, const int32_t* seqlens_k,
                        double scale, double* o, double* lse) {
    int rc = check_args(q, k, v, kind, B, H, Nq, Nk, d);
    if (rc) return rc;
    if (!o || !lse) return -1;
    Decoded x;
    if (decode_inputs(q, k, v, NULL, kind, B * Nq * H * d, B * Nk * H * d, &x)) return -4;
    const int64_t rows = B * H * Nq;
    int failed = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc((size_t)Nk * sizeof(double));
        if (!s) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < rows; ++r) {
                /* r enumerates (b, h, i) with i fastest */
                const int64_t i = r % Nq, h = (r / Nq) % H, b = r / (Nq * H);
                int64_t lo, hi;
                key_range(i + Nk - Nq, causal, window_left, window_right,
                          batch_key_length(seqlens_k, b, Nk), &lo, &hi);
                attention_row(x.q, x.k, x.v, Nq, Nk, H, d, lo, hi, scale, b, h, i, s,
                              o + ((b * Nq + i) * H + h) * d, lse + (b * H + h) * Nq + i);
            }
            free(s);
        }
    }
    release(&x);
    return failed ? -4 : 0;
}

int oracle_attention_masked(const void* q, const void* k, const void* v, int kind, int64_t B,
                            int64_t H, int64_t N, int64_t d, int causal, int64_t window_left,
                            int64_t window_right, const int32_t* seqlens_k, double scale,
                            double* o, double* lse) {
    return oracle_attention_qk(q, k, v, kind, B, H, N, N, d, causal, window_left, window_right,
                               seqlens_k, scale, o, lse);
}

int oracle_attention(const void* q, const void* k, const void* v, int kind, int64_t B,
                     int64_t H, int64_t N, int64_t d, int causal, double scale, double* o,
                     double* lse) {
    return oracle_attention_qk(q, k, v, kind, B, H, N, N, d, causal, -1, -1, 0, scale, o, lse);
}

/* Selected rows: rows[3t..3t+2] = (b, h, i); o_rows [nrows, d], lse_rows [nrows]. */
int oracle_attention_rows_qk(const void* q, const void* k, const void* v, int kind, int64_t B,
                             int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal,
                             int64_t window_left, int64_t window_right,
                             const int32_t* seqlens_k, double scale, const int64_t* rows,
                             int64_t nrows, double* o_rows, double* lse_rows) {
    int rc = check_args(q, k, v, kind, B, H, Nq, Nk, d);
    if (rc) return rc;
    if (!rows || !o_rows || !lse_rows || nrows < 0) return -1;
    for (int64_t t = 0; t < nrows; ++t) {
        const int64_t b = rows[3 * t], h = rows[3 * t + 1], i = rows[3 * t + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= Nq) return -5;
    }
    Decoded x;
    if (decode_inputs(q, k, v, NULL, kind, B * Nq * H * d, B * Nk * H * d, &x)) return -4;
    int failed = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc((size_t)Nk * sizeof(double));
        if (!s) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < nrows; ++t) {
                const int64_t b = rows[3 * t], h = rows[3 * t + 1], i = rows[3 * t + 2];
                int64_t lo, hi;
                key_range(i + Nk - Nq, causal, window_left, window_right,
                          batch_key_length(seqlens_k, b, Nk), &lo, &hi);
                attention_row(x.q, x.k, x.v, Nq, Nk, H, d, lo, hi, scale, b, h, i, s,
                              o_rows + t * d, lse_rows + t);
            }
            free(s);
        }
    }
    release(&x);
    return failed ? -4 : 0;
}

int oracle_attention_rows_masked(const void* q, const void* k, const void* v, int kind,
                                 int64_t B, int64_t H, int64_t N, int64_t d, int causal,
                                 int64_t window_left, int64_t window_right,
                                 const int32_t* seqlens_k, double scale, const int64_t* rows,
                                 int64_t nrows, double* o_rows, double* lse_rows) {
    return oracle_attention_rows_qk(q, k, v, kind, B, H, N, N, d, causal, window_left,
                                    window_right, seqlens_k, scale, rows, nrows, o_rows,
                                    lse_rows);
}

int oracle_attention_rows(const void* q, const void* k, const void* v, int kind, int64_t B,
                          int64_t H, int64_t N, int64_t d, int causal, double scale,
                          const int64_t* rows, int64_t nrows, double* o_rows,
                          double* lse_rows) {
    return oracle_attention_rows_qk(q, k, v, kind, B, H, N, N, d, causal, -1, -1, 0, scale,
                                    rows, nrows, o_rows, lse_rows);
}

/*
 * The same backward on sampled outputs, for sizes where the N x N matrices of
 * oracle_attention_bwd do not fit in memory. The formulas are those of oracle_attention_bwd,
 * evaluated element by element. For each sampled head (b, h) = (heads[2t], heads[2t+1]):
 *   1. for every query i: the row maximum m_i and sum l_i of the forward's softmax (two passes
 *      over the allowed keys), and D_i = sum_j P_ij dP_ij with P_ij = exp(s_ij - m_i) / l_i,
 *      s_ij = scale <q_i, k_j>, dP_ij = <dO_i, v_j>;
 *   2. for each sampled key j: dV_j = sum_i P_ij dO_i and dK_j = scale sum_i dS_ij q_i with
 *      dS_ij = P_ij (dP_ij - D_i), over the queries i that see key j;
 *   3. for each sampled query i: dQ_i = scale sum_j dS_ij k_j over the keys it sees.
 * Masks: causal or none (queries and keys share N). Outputs (fp64, row-major):
 * dq [nheads][nqueries][d], dk and dv [nheads][nkeys][d].
 */
int oracle_attention_bwd_sampled(const void* q, const void* k, const void* v, const void* dout,
                                 int kind, int64_t B, int64_t H, int64_t N, int64_t d,
                                 int causal, int64_t window_left, int64_t window_right,
                                 const int32_t* seqlens_k, double scale, const int64_t* heads,
                                 int64_t nheads, const int64_t* keys, int64_t nkeys,
                                 const int64_t* queries, int64_t nqueries, double* dq, double* dk,
                                 double* dv) {
    int rc = check_args(q, k, v, kind, B, H, N, N, d);
    if (rc) return rc;
    if (!dout || !heads || nheads < 0 || nkeys < 0 || nqueries < 0) return -1;
    if ((nkeys && (!keys || !dk || !dv)) || (nqueries && (!queries || !dq))) return -1;
    for (int64_t t = 0; t < nheads; ++t)
        if (heads[2 * t] < 0 || heads[2 * t] >= B || heads[2 * t + 1] < 0 ||
            heads[2 * t + 1] >= H) return -2;
    for (int64_t t = 0; t < nkeys; ++t) if (keys[t] < 0 || keys[t] >= N) return -2;
    for (int64_t t = 0; t < nqueries; ++t) if (queries[t] < 0 || queries[t] >= N) return -2;
    Decoded x;
    if (decode_inputs(q, k, v, dout, kind, B * N * H * d, B * N * H * d, &x)) return -4;
    const double *qd = x.q, *kd = x.k, *vd = x.v, *gd = x.g;
    double* m = (double*)malloc((size_t)N * sizeof(double));
    double* l = (double*)malloc((size_t)N * sizeof(double));
    double* D = (double*)malloc((size_t)N * sizeof(double));
    if (!m || !l || !D) {
        free(m);
        free(l);
        free(D);
        release(&x);
        return -4;
    }
    for (int64_t t = 0; t < nheads; ++t) {
        const int64_t b = heads[2 * t], h = heads[2 * t + 1];
        const int64_t len_b = batch_key_length(seqlens_k, b, N);
#define ROW(i) ((((b) * N + (i)) * H + (h)) * d)
        /* 1. row statistics of every query of this head, over its allowed keys [lo, hi) */
#pragma omp parallel for schedule(dynamic, 16)
        for (int64_t i = 0; i < N; ++i) {
            int64_t lo, hi;
            key_range(i, causal, window_left, window_right, len_b, &lo, &hi);
            double mi = -INFINITY;
            for (int64_t j = lo; j < hi; ++j) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += qd[ROW(i) + c] * kd[ROW(j) + c];
                if (scale * dot > mi) mi = scale * dot;
            }
            double li = 0.0, di = 0.0;
            for (int64_t j = lo; j < hi; ++j) {
                double dot = 0.0, dp = 0.0;
                for (int64_t c = 0; c < d; ++c) {
                    dot += qd[ROW(i) + c] * kd[ROW(j) + c];
                    dp += gd[ROW(i) + c] * vd[ROW(j) + c];
                }
                const double e = exp(scale * dot - mi);
                li += e;
                di += e * dp;
            }
            m[i] = mi;
            l[i] = li;
            D[i] = li > 0.0 ? di / li : 0.0;
        }
        /* 2. dV_j, dK_j for the sampled keys: every query whose allowed range holds key j */
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t u = 0; u < nkeys; ++u) {
            const int64_t j = keys[u];
            double* gk = dk + (t * nkeys + u) * d;
            double* gv = dv + (t * nkeys + u) * d;
            for (int64_t c = 0; c < d; ++c) gk[c] = gv[c] = 0.0;
            for (int64_t i = 0; i < N; ++i) {
                int64_t lo, hi;
                key_range(i, causal, window_left, window_right, len_b, &lo, &hi);
                if (j < lo || j >= hi) continue;
                double dot = 0.0, dp = 0.0;
                for (int64_t c = 0; c < d; ++c) {
                    dot += qd[ROW(i) + c] * kd[ROW(j) + c];
                    dp += gd[ROW(i) + c] * vd[ROW(j) + c];
                }
                const double p = exp(scale * dot - m[i]) / l[i];
                const double ds = p * (dp - D[i]);
                for (int64_t c = 0; c < d; ++c) {
                    gv[c] += p * gd[ROW(i) + c];
                    gk[c] += ds * qd[ROW(i) + c];
                }
            }
            for (int64_t c = 0; c < d; ++c) gk[c] *= scale;
        }
        /* 3. dQ_i for the sampled queries, over their allowed keys */
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t u = 0; u < nqueries; ++u) {
            const int64_t i = queries[u];
            double* gq = dq + (t * nqueries + u) * d;
            for (int64_t c = 0; c < d; ++c) gq[c] = 0.0;
            int64_t lo, hi;
            key_range(i, causal, window_left, window_right, len_b, &lo, &hi);
            for (int64_t j = lo; j < hi; ++j) {
                double dot = 0.0, dp = 0.0;
                for (int64_t c = 0; c < d; ++c) {
                    dot += qd[ROW(i) + c] * kd[ROW(j) + c];
                    dp += gd[ROW(i) + c] * vd[ROW(j) + c];
                }
                const double ds = exp(scale * dot - m[i]) / l[i] * (dp - D[i]);
                for (int64_t c = 0; c < d; ++c) gq[c] += ds * kd[ROW(j) + c];
            }
            for (int64_t c = 0; c < d; ++c) gq[c] *= scale;
        }
#undef ROW
    }
    free(m);
    free(l);
    free(D);
    release(&x);
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Backward of the same attention (the gradients the kept statistics serve: "FlashAttention
 * V2 核心原理与架构设计" §2.3 keeps m and l for the backward pass). With L = sum dO . O for a given
 * upstream gradient dO, the chain rule through S = scale Q K^T, P = softmax(S), O = P V gives
 *   dV = P^T dO,   dP = dO V^T,   dS_ij = P_ij (dP_ij - D_i) with D_i = sum_j P_ij dP_ij,
 *   dQ = scale dS K,   dK = scale dS^T Q.
 * Keys outside a query's allowed interval have P_ij = 0 (so dS_ij = 0). Queries and keys share
 * N here. Per (b, h) the N x N matrix P is materialised in fp64; no blocking. Layouts as the
 * forward: q, k, v, dout and dq, dk, dv are [B, N, H, d].
 */
int oracle_attention_bwd(const void* q, const void* k, const void* v, const void* dout,
                         int kind, int64_t B, int64_t H, int64_t N, int64_t d, int causal,
                         int64_t window_left, int64_t window_right, const int32_t* seqlens_k,
                         double scale, double* dq, double* dk, double* dv) {
    int rc = check_args(q, k, v, kind, B, H, N, N, d);
    if (rc) return rc;
    if (!dout || !dq || !dk || !dv) return -1;
    Decoded x;
    if (decode_inputs(q, k, v, dout, kind, B * N * H * d, B * N * H * d, &x)) return -4;
    const double *qd = x.q, *kd = x.k, *vd = x.v, *gd = x.g;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const int64_t b = bh / H, h = bh % H;
        double* P = (double*)calloc((size_t)(N * N), sizeof(double));
        double* dS = (double*)calloc((size_t)(N * N), sizeof(double));
        if (!P || !dS) {
            free(P);
            free(dS);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        const int64_t len_b = batch_key_length(seqlens_k, b, N);
        /* P, row by row (three-pass softmax over the allowed keys) */
        for (int64_t i = 0; i < N; ++i) {
            int64_t lo, hi;
            key_range(i, causal, window_left, window_right, len_b, &lo, &hi);
            if (lo >= hi) continue;
            const int64_t q_off = ((b * N + i) * H + h) * d;
            double m = -INFINITY;
            for (int64_t j = lo; j < hi; ++j) {
                const int64_t k_off = ((b * N + j) * H + h) * d;
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += qd[q_off + c] * kd[k_off + c];
                P[i * N + j] = scale * dot;
                if (P[i * N + j] > m) m = P[i * N + j];
            }
            double l = 0.0;
            for (int64_t j = lo; j < hi; ++j) l += exp(P[i * N + j] - m);
            for (int64_t j = lo; j < hi; ++j) P[i * N + j] = exp(P[i * N + j] - m) / l;
        }
        /* dP = dO V^T, D_i = sum_j P_ij dP_ij, dS = P (dP - D) */
        for (int64_t i = 0; i < N; ++i) {
            const int64_t o_off = ((b * N + i) * H + h) * d;
            double Di = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                if (P[i * N + j] == 0.0) continue;
                const int64_t v_off = ((b * N + j) * H + h) * d;
                double dp = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dp += gd[o_off + c] * vd[v_off + c];
                dS[i * N + j] = dp;
                Di += P[i * N + j] * dp;
            }
            for (int64_t j = 0; j < N; ++j) dS[i * N + j] = P[i * N + j] * (dS[i * N + j] - Di);
        }
        /* dQ = scale dS K */
        for (int64_t i = 0; i < N; ++i) {
            double* out = dq + ((b * N + i) * H + h) * d;
            for (int64_t c = 0; c < d; ++c) out[c] = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                if (dS[i * N + j] == 0.0) continue;
                const int64_t k_off = ((b * N + j) * H + h) * d;
                for (int64_t c = 0; c < d; ++c) out[c] += dS[i * N + j] * kd[k_off + c];
            }
            for (int64_t c = 0; c < d; ++c) out[c] *= scale;
        }
        /* dK = scale dS^T Q, dV = P^T dO */
        for (int64_t j = 0; j < N; ++j) {
            double* gk = dk + ((b * N + j) * H + h) * d;
            double* gv = dv + ((b * N + j) * H + h) * d;
            for (int64_t c = 0; c < d; ++c) gk[c] = gv[c] = 0.0;
            for (int64_t i = 0; i < N; ++i) {
                const int64_t row = ((b * N + i) * H + h) * d;
                const double ds = dS[i * N + j], p = P[i * N + j];
                if (ds != 0.0)
                    for (int64_t c = 0; c < d; ++c) gk[c] += ds * qd[row + c];
                if (p != 0.0)
                    for (int64_t c = 0; c < d; ++c) gv[c] += p * gd[row + c];
            }
            for (int64_t c = 0; c < d; ++c) gk[c] *= scale;
        }
        free(P);
        free(dS);
    }
    release(&x);
    return failed ? -4 : 0;
}
