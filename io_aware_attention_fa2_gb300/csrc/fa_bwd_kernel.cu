// fa_bwd_kernel.cu -- attention backward for sm_103a: dQ, dK, dV from Q, K, V, O, dO and the
// forward's LSE, with tcgen05 MMAs accumulating in TMEM.
//
// The statistics the forward keeps ("FlashAttention V2 核心原理与架构设计" §2.3: l and m, kept
// here as LSE = m + ln l) let the backward rebuild P exactly without a second softmax pass:
// P_ij = exp(scale <q_i, k_j> - LSE_i). With D_i = <dO_i, O_i> (= sum_j P_ij dP_ij), the
// chain rule through softmax gives
//   dV = P^T dO,  dP = dO V^T,  dS' = scale * P (dP - D),  dK = dS'^T Q,  dQ = dS' K.
//
// Work split: one CTA per (b, h, K/V block j of 128 keys); K_j, V_j stay in shared memory and
// dK_j, dV_j accumulate in TMEM while the CTA walks the Q blocks i that can see block j (all of
// them, or i >= j when causal: the FA2 loop order with the roles of the two operands swapped).
// Each step's dQ_i contribution is added to an fp32 workspace with vector reductions; a
// pre-kernel computes D and clears the workspace, a post-kernel rounds dQ.
//
// Per step (Q block i), all MMAs M = 128, fp32 accumulators in TMEM:
//   S^T  = K_j Q_i^T     (smem x smem)            -> T_S   lanes = keys, columns = queries
//   dP^T = V_j dO_i^T    (smem x smem)            -> T_dP
//   compute warps: P^T = exp2(S^T scale log2e - LSE_i log2e) (masked), written back over T_S
//                  as 16-bit pairs; dS'^T = scale P^T (dP^T - D_i), written over T_dP and, as
//                  rows of dS'^T (queries contiguous), into shared memory
//   dV  += P^T dO_i      (TMEM x smem, dO MN-major)
//   dK  += dS'^T Q_i     (TMEM x smem, Q MN-major)
//   dQ_i = dS' K_j       (smem x smem: dS' M-major, K MN-major) -> T_dP, lanes = queries
//   dQ warps: dQ_i rows -> fp32 workspace (red.global.add.v4.f32)
// MMA issue order: dV(i), S^T(i+1), dK(i), dQ(i), dP^T(i+1): the next S^T runs while the
// softmax warps compute dS'(i), and the next dP^T waits only for dQ(i) to be read out.
// TMEM columns: T_S [0,128), T_dP [128,256), dV [256, 256+d), dK [256+d, 256+2d).
//
// Warps: 0 TMA producer (K_j, V_j once; Q_i, dO_i into a 2-deep ring), 1 MMA issuer and TMEM
// allocator, 2..5 softmax / dS' (thread <-> TMEM lane), 6..9 dQ read-out and reduction.
// Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "ptx_sm103.cuh"

namespace fa {

// Error word of the backward kernels (the forward has its own): nonzero after a wait ran out.
__device__ int g_bwd_device_error = 0;

namespace {

constexpr int kBwdThreads = 320;   // producer, MMA, 4 softmax / dS' warps, 4 dQ warps
constexpr int kBwdStages = 2;
constexpr uint32_t kBoxBytes = BOX_ROWS * BOX_COLS * 2;   // 16 KiB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kT_S = 0, kT_dP = 128, kT_dV = 256;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kErrTimeout = -8;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdSmem {
  static constexpr uint32_t kTile = (D / BOX_COLS) * kBoxBytes;   // 128 rows x d
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kTile;
  static constexpr uint32_t kQ = kV + kTile;                      // + stage * kTile
  static constexpr uint32_t kdO = kQ + kBwdStages * kTile;        // + stage * kTile
  static constexpr uint32_t kdS = kdO + kBwdStages * kTile;       // 128 keys x 128 queries
  static constexpr uint32_t kStat = kdS + 2 * kBoxBytes;   // [LSE*log2e, D][128]
  static constexpr uint32_t kBars = kStat + 2 * 128 * 4;
  static constexpr uint32_t kEnd = kBars + 16 * 8;
  static constexpr uint32_t kDynamic = kEnd + 1024;
};

enum : int {
  BB_KV_FULL = 0,
  BB_QD_FULL = 1,                          // + stage
  BB_QD_EMPTY = BB_QD_FULL + kBwdStages,   // + stage
  BB_S_FULL = BB_QD_EMPTY + kBwdStages,    // S^T computed
  BB_DP_FULL,                              // dP^T computed
  BB_P_FULL,                               // P^T in TMEM (128 arrivals)
  BB_DS_FULL,                              // dS'^T in TMEM and shared memory (128 arrivals)
  BB_DQ_FULL,                              // dQ_i in TMEM (T_dP; this step's dV, dK done)
  BB_DQ_TAKEN,                             // dQ_i read out of TMEM (128 arrivals)
  BB_STAT,                                 // this step's LSE, D in shared memory (128)
  BB_MMA_DONE,
  BB_COUNT
};
static_assert(BB_COUNT <= 16, "barrier slots");

__device__ __forceinline__ void record_timeout(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(&g_bwd_device_error, 0, kErrTimeout);
}

template <bool FP16>
__device__ __forceinline__ float load_elem(const void* p, int64_t i) {
  if constexpr (FP16) return __half2float(static_cast<const __half*>(p)[i]);
  else return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

template <bool FP16>
__device__ __forceinline__ void unpack2(uint32_t w, float& lo, float& hi) {
  if constexpr (FP16) {
    const __half2 h = *reinterpret_cast<const __half2*>(&w);
    lo = __low2float(h);
    hi = __high2float(h);
  } else {
    // a bf16 value is the upper half of the fp32 with the same bits
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  }
}

template <bool FP16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (FP16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// D[b, h, q] = <dO[b, q, h, :], O[b, q, h, :]> and dQ workspace rows cleared. One warp per
// (b, q, h) row of the [B, N, H, d] tensors.
template <int D, bool FP16>
__global__ void __launch_bounds__(256)
    fa_bwd_pre_kernel(const void* __restrict__ o, const void* __restrict__ dout,
                      float* __restrict__ dpre, float* __restrict__ dq_acc, int H, int N,
                      long long rows) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32;
  if (row >= rows) return;
  const int lane = threadIdx.x % 32;
  float acc = 0.f;
#pragma unroll
  for (int c = lane; c < D; c += 32)
    acc = fmaf(load_elem<FP16>(o, row * D + c), load_elem<FP16>(dout, row * D + c), acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  float4* z = reinterpret_cast<float4*>(dq_acc + row * D);
  for (int c = lane; c < D / 4; c += 32) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (lane == 0) {
    const long long h = row % H, bq = row / H;   // row = (b * N + q) * H + h
    const long long q = bq % N, b = bq / N;
    dpre[(b * H + h) * N + q] = acc;
  }
}

// dQ (input type) from the fp32 workspace, element-wise.
template <bool FP16>
__global__ void __launch_bounds__(256)
    fa_bwd_post_kernel(const float* __restrict__ dq_acc, void* __restrict__ dq,
                       long long pairs) {
  const long long t = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (t >= pairs) return;
  const float2 v = reinterpret_cast<const float2*>(dq_acc)[t];
  static_cast<uint32_t*>(dq)[t] = pack2<FP16>(v.x, v.y);
}

// ---------------------------------------------------------------------------------------------
template <int D, bool FP16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_do, const float* __restrict__ lse,
                  const float* __restrict__ dpre, float* __restrict__ dq_acc,
                  void* __restrict__ dk_ptr, void* __restrict__ dv_ptr, int H, int N, int causal,
                  float scale, float scale_log2) {
  using L = BwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  const uint32_t smem_base = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* const smem_gen = smem_raw + (smem_base - ptx::smem_addr(smem_raw));
  const uint32_t sK = smem_base + L::kK, sV = smem_base + L::kV;
  const uint32_t sQ = smem_base + L::kQ, sdO = smem_base + L::kdO, sdS = smem_base + L::kdS;
  float* const stat = reinterpret_cast<float*>(smem_gen + L::kStat);   // [2][128]
  static_assert(BwdSmem<D>::kDynamic <= 227 * 1024, "backward tiles exceed shared memory");
  auto bar = [&](int i) { return smem_base + L::kBars + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Unit: (b, h) x K/V block; blocks of one head are consecutive, longest (causal) first.
  const int num_kv = (N + BLOCK_N - 1) / BLOCK_N;
  const int num_q = (N + BLOCK_M - 1) / BLOCK_M;
  const int bh = static_cast<int>(blockIdx.x) / num_kv;
  const int rj = static_cast<int>(blockIdx.x) % num_kv;
  const int jb = rj;                                     // K/V block (block 0 sees most Q)
  const int b = bh / H, h = bh % H;
  const int i0 = causal ? jb : 0;                        // first Q block that sees block jb
  const int steps = num_q - i0;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(bar(BB_KV_FULL), 1);
    for (int s = 0; s < kBwdStages; ++s) {
      ptx::mbar_init(bar(BB_QD_FULL + s), 1);
      ptx::mbar_init(bar(BB_QD_EMPTY + s), 1);
    }
    ptx::mbar_init(bar(BB_S_FULL), 1);
    ptx::mbar_init(bar(BB_DP_FULL), 1);
    ptx::mbar_init(bar(BB_P_FULL), 128);
    ptx::mbar_init(bar(BB_DS_FULL), 128);
    ptx::mbar_init(bar(BB_DQ_FULL), 1);
    ptx::mbar_init(bar(BB_DQ_TAKEN), 128);
    ptx::mbar_init(bar(BB_STAT), 128);
    ptx::mbar_init(bar(BB_MMA_DONE), 1);
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&tmem_base_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = tmem_base_slot;
  volatile int* abort_p = &abort_flag;
  auto wait = [&](int slot, uint32_t parity) {
    return ptx::wait_bounded(bar(slot), parity, abort_p, kWaitLimitNs);
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tm_q);
      ptx::prefetch_tensormap(&tm_k);
      ptx::prefetch_tensormap(&tm_v);
      ptx::prefetch_tensormap(&tm_do);
      ptx::mbar_arrive_expect_tx(bar(BB_KV_FULL), 2 * L::kTile);
      for (int c = 0; c < D / BOX_COLS; ++c) {
        ptx::tma_load_4d(sK + c * kBoxBytes, &tm_k, bar(BB_KV_FULL), c * BOX_COLS, h,
                         jb * BLOCK_N, b);
        ptx::tma_load_4d(sV + c * kBoxBytes, &tm_v, bar(BB_KV_FULL), c * BOX_COLS, h,
                         jb * BLOCK_N, b);
      }
      int issued = 0;
      for (int n = 0; n < steps; ++n) {
        const int s = n % kBwdStages;
        if (!wait(BB_QD_EMPTY + s, ((n / kBwdStages) & 1) ^ 1)) {
          record_timeout(abort_p);
          break;
        }
        const int q_row0 = (i0 + n) * BLOCK_M;
        ptx::mbar_arrive_expect_tx(bar(BB_QD_FULL + s), 2 * L::kTile);
        for (int c = 0; c < D / BOX_COLS; ++c) {
          ptx::tma_load_4d(sQ + s * L::kTile + c * kBoxBytes, &tm_q, bar(BB_QD_FULL + s),
                           c * BOX_COLS, h, q_row0, b);
          ptx::tma_load_4d(sdO + s * L::kTile + c * kBoxBytes, &tm_do, bar(BB_QD_FULL + s),
                           c * BOX_COLS, h, q_row0, b);
        }
        issued = n + 1;
      }
      wait(BB_KV_FULL, 0);
      for (int n = (issued > kBwdStages ? issued - kBwdStages : 0); n < issued; ++n)
        wait(BB_QD_FULL + n % kBwdStages, (n / kBwdStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_st = ptx::idesc_f16(FP16, 128, BLOCK_M, false);         // S^T, dP^T
      constexpr uint32_t id_acc = ptx::idesc_f16(FP16, 128, D, true);               // dV, dK
      constexpr uint32_t id_dq = ptx::idesc_f16(FP16, BLOCK_M, D, true, true);      // dQ
      auto qbase = [&](int n) { return sQ + (n % kBwdStages) * L::kTile; };
      auto dobase = [&](int n) { return sdO + (n % kBwdStages) * L::kTile; };
      // S^T = K_j Q_i^T -> T_S and dP^T = V_j dO_i^T -> T_dP: both operands K-major over d.
      auto issue_s = [&](int n) {
        ptx::tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * kBoxBytes + (kk % 4) * 32;
          ptx::mma_f16_ss(tmem + kT_S, ptx::smem_desc_sw128(sK + off, 16, 1024),
                          ptx::smem_desc_sw128(qbase(n) + off, 16, 1024), id_st, kk > 0);
        }
        ptx::mma_commit(bar(BB_S_FULL));
      };
      auto issue_dp = [&](int n) {
        ptx::tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * kBoxBytes + (kk % 4) * 32;
          ptx::mma_f16_ss(tmem + kT_dP, ptx::smem_desc_sw128(sV + off, 16, 1024),
                          ptx::smem_desc_sw128(dobase(n) + off, 16, 1024), id_st, kk > 0);
        }
        ptx::mma_commit(bar(BB_DP_FULL));
      };
      bool ok = wait(BB_KV_FULL, 0) && wait(BB_QD_FULL + 0, 0);
      if (ok) {
        issue_s(0);
        issue_dp(0);
      }
      for (int n = 0; ok && n < steps; ++n) {
        const int s = n % kBwdStages;
        const bool next = n + 1 < steps;
        // dV += P^T dO_i: A = P^T from TMEM (16 queries = 8 columns per MMA); B = dO_i with
        // d contiguous (MN-major): 16 query rows of 128 bytes per MMA, LBO = next 64 columns.
        if (!wait(BB_P_FULL, n & 1)) { ok = false; break; }
        ptx::tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < BLOCK_M / 16; ++kk)
          ptx::mma_f16_ts(tmem + kT_dV, tmem + kT_S + kk * 8,
                          ptx::smem_desc_sw128(dobase(n) + kk * 16 * 128, kBoxBytes, 1024),
                          id_acc, (n > 0 || kk > 0) ? 1u : 0u);
        // S^T(i+1) over P^T(i): issued after dV(i), which reads P^T first (in-order pipe).
        if (next) {
          if (!wait(BB_QD_FULL + (n + 1) % kBwdStages, ((n + 1) / kBwdStages) & 1)) {
            ok = false;
            break;
          }
          issue_s(n + 1);
        }
        // dK += dS'^T Q_i, same shapes with Q_i as B.
        if (!wait(BB_DS_FULL, n & 1)) { ok = false; break; }
        ptx::tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < BLOCK_M / 16; ++kk)
          ptx::mma_f16_ts(tmem + kT_dV + D, tmem + kT_dP + kk * 8,
                          ptx::smem_desc_sw128(qbase(n) + kk * 16 * 128, kBoxBytes, 1024),
                          id_acc, (n > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(bar(BB_QD_EMPTY + s));   // Q_i and dO_i are no longer read
        // dQ_i = dS' K_j -> T_dP (after dK has read dS'^T there): A = dS' (queries contiguous,
        // M-major) from shared memory, B = K_j (d contiguous, MN-major); 16 keys = 16 rows of
        // 128 bytes per MMA for both.
#pragma unroll
        for (int kk = 0; kk < BLOCK_N / 16; ++kk)
          ptx::mma_f16_ss(tmem + kT_dP,
                          ptx::smem_desc_sw128(sdS + kk * 16 * 128, kBoxBytes, 1024),
                          ptx::smem_desc_sw128(sK + kk * 16 * 128, kBoxBytes, 1024), id_dq,
                          kk > 0);
        ptx::mma_commit(bar(BB_DQ_FULL));
        // dP^T(i+1) over dQ(i) once the dQ warps have read it out.
        if (next) {
          if (!wait(BB_DQ_TAKEN, n & 1)) { ok = false; break; }
          issue_dp(n + 1);
        }
      }
      if (!ok) record_timeout(abort_p);
      ptx::mma_commit(bar(BB_MMA_DONE));
      wait(BB_MMA_DONE, 0);
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;                 // TMEM lanes [32q, 32q+32)
    const int r = quarter * 32 + lane;            // TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    if (warp < 6) {
      // -------------------------------------------------------------- softmax / dS' warps
      // lane r = key jb * 128 + r for S^T, dP^T, dV, dK
      const int key = jb * BLOCK_N + r;
      const bool key_ok = key < N;
      uint8_t* const ds_gen = smem_gen + L::kdS;
      for (int n = 0; n < steps; ++n) {
        const int q0 = (i0 + n) * BLOCK_M;
        float* const s_lse = stat;         // LSE_i * log2e, +inf for rows to ignore
        float* const s_d = stat + 128;     // D_i
        {
          // This step's row statistics, one query per thread. Queries past N (and rows with
          // no allowed key, LSE = -inf) get +inf, so their P is 0. One buffer serves every
          // step: it is overwritten only after all 128 threads have finished the previous
          // step's dS' (DS_FULL), the last phase that reads it.
          const int q = q0 + r;
          float l2 = INFINITY, dd = 0.f;
          if (q < N) {
            const float lv = lse[static_cast<int64_t>(bh) * N + q];
            if (lv != -INFINITY) l2 = lv * kLog2e;
            dd = dpre[static_cast<int64_t>(bh) * N + q];
          }
          if (n > 0 && !wait(BB_DS_FULL, (n - 1) & 1)) { ok = false; break; }
          s_lse[r] = l2;
          s_d[r] = dd;
          ptx::mbar_arrive(bar(BB_STAT));
          if (!wait(BB_STAT, n & 1)) { ok = false; break; }
        }
        // --- P^T: this thread's key against the 128 queries of block i
        if (!wait(BB_S_FULL, n & 1)) { ok = false; break; }
        ptx::tc_fence_after_sync();
      // P^T, kept packed as 16-bit pairs (the values the dV product uses, also used for dS'):
        // query q0 + t sees this key only if key <= q0 + t (causal); keys past N do not exist.
        const int lim = !key_ok ? BLOCK_M : (causal ? min(max(key - q0, 0), BLOCK_M) : 0);
        uint32_t pp[BLOCK_M / 2];
#pragma unroll
        for (int c = 0; c < BLOCK_M / 32; ++c) {
          uint32_t sr[32];
          ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_S + c * 32, sr);
          ptx::tmem_wait_ld();
          ptx::reg_fence(sr);
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int a = 32 * c + 2 * t;
            float p0 = ptx::exp2_approx(fmaf(__uint_as_float(sr[2 * t]), scale_log2, -s_lse[a]));
            float p1 = ptx::exp2_approx(
                fmaf(__uint_as_float(sr[2 * t + 1]), scale_log2, -s_lse[a + 1]));
            if (a < lim) p0 = 0.f;
            if (a + 1 < lim) p1 = 0.f;
            pp[16 * c + t] = pack2<FP16>(p0, p1);
          }
          uint32_t pr[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) pr[t] = pp[16 * c + t];
          ptx::tmem_st_32x32b_x16(tmem + lane_off + kT_S + c * 16, pr);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before_sync();
        ptx::mbar_arrive(bar(BB_P_FULL));

        // --- dS'^T = scale P^T (dP^T - D) -> TMEM (over dP^T) and shared memory (rows of dS'^T).
        // dP^T(i) was issued after dQ(i-1) completed, so shared dS' is free again.
        if (!wait(BB_DP_FULL, n & 1)) { ok = false; break; }
        ptx::tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < BLOCK_M / 32; ++c) {
          uint32_t dr[32];
          ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_dP + c * 32, dr);
          ptx::tmem_wait_ld();
          ptx::reg_fence(dr);
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int a = 32 * c + 2 * t;
            float p0, p1;
            unpack2<FP16>(pp[16 * c + t], p0, p1);
            const float d0 = scale * p0 * (__uint_as_float(dr[2 * t]) - s_d[a]);
            const float d1 = scale * p1 * (__uint_as_float(dr[2 * t + 1]) - s_d[a + 1]);
            pk[t] = pack2<FP16>(d0, d1);
          }
          ptx::tmem_st_32x32b_x16(tmem + lane_off + kT_dP + c * 16, pk);
          // queries 32c .. 32c+31 of key row r: 4 chunks of 16 bytes in box c / 2, swizzled
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int chunk = (c % 2) * 4 + u;        // 16-byte chunk within the 128-byte row
            const uint32_t off = (c / 2) * kBoxBytes + r * 128 + ((chunk ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(ds_gen + off) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        }
        ptx::tmem_wait_st();
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before_sync();
        ptx::mbar_arrive(bar(BB_DS_FULL));

      }
      if (ok) {
        // dK, dV rows. The last dQ completion implies this CTA's MMAs are all complete.
        if (!wait(BB_DQ_FULL, (steps - 1) & 1)) ok = false;
      }
      if (ok) {
        ptx::tc_fence_after_sync();
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          uint16_t* out = static_cast<uint16_t*>(which ? dk_ptr : dv_ptr) +
                          ((static_cast<int64_t>(b) * N + key) * H + h) * D;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t gr[32];
            ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_dV + which * D + c * 32, gr);
            ptx::tmem_wait_ld();
            ptx::reg_fence(gr);
            if (key_ok) {
              uint4* dst = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
              for (int t = 0; t < 4; ++t)
                dst[t] = make_uint4(
                    pack2<FP16>(__uint_as_float(gr[8 * t]), __uint_as_float(gr[8 * t + 1])),
                    pack2<FP16>(__uint_as_float(gr[8 * t + 2]), __uint_as_float(gr[8 * t + 3])),
                    pack2<FP16>(__uint_as_float(gr[8 * t + 4]), __uint_as_float(gr[8 * t + 5])),
                    pack2<FP16>(__uint_as_float(gr[8 * t + 6]), __uint_as_float(gr[8 * t + 7])));
            }
          }
        }
      } else {
        record_timeout(abort_p);
      }
    } else {
      // -------------------------------------------------------------- dQ warps
      // lane r = query q0 + r of dQ_i (in T_dP); its row goes into the fp32 workspace.
      for (int n = 0; n < steps; ++n) {
        const int q0 = (i0 + n) * BLOCK_M;
        if (!wait(BB_DQ_FULL, n & 1)) { ok = false; break; }
        ptx::tc_fence_after_sync();
        // 32 columns at a time: the reductions of one chunk overlap the next chunk's load;
        // T_dP is released as soon as the last chunk is in registers.
        const bool row_ok = q0 + r < N;
        float* dst = dq_acc + ((static_cast<int64_t>(b) * N + q0 + r) * H + h) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t qr[32];
          ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_dP + c * 32, qr);
          ptx::tmem_wait_ld();
          ptx::reg_fence(qr);
          if (c == D / 32 - 1) {
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(bar(BB_DQ_TAKEN));
          }
          if (row_ok) {
#pragma unroll
            for (int t = 0; t < 32; t += 4)
              ptx::red_add_v4(dst + c * 32 + t, __uint_as_float(qr[t]), __uint_as_float(qr[t + 1]),
                              __uint_as_float(qr[t + 2]), __uint_as_float(qr[t + 3]));
          }
        }
      }
      if (!ok) record_timeout(abort_p);
    }
  }

  // ------------------------------------------------------------------ teardown
  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool FP16>
cudaError_t launch_bwd_impl(const BwdParams& p, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.B) * p.N * p.H;
  fa_bwd_pre_kernel<D, FP16><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
      p.o, p.dout, p.dpre, p.dq_acc, p.H, p.N, rows);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  auto kernel = fa_bwd_kernel<D, FP16>;
  const size_t smem = BwdSmem<D>::kDynamic;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const long long num_kv = (p.N + BLOCK_N - 1) / BLOCK_N;
  kernel<<<static_cast<unsigned>(num_kv * p.B * p.H), kBwdThreads, smem, stream>>>(
      p.tm_q, p.tm_k, p.tm_v, p.tm_do, p.lse, p.dpre, p.dq_acc, p.dk, p.dv, p.H, p.N, p.causal,
      p.scale, p.scale * kLog2e);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const long long pairs = rows * D / 2;
  fa_bwd_post_kernel<FP16><<<static_cast<unsigned>((pairs + 255) / 256), 256, 0, stream>>>(
      p.dq_acc, p.dq, pairs);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_smem_bytes(int d) {
  return d == 64 ? BwdSmem<64>::kDynamic : BwdSmem<128>::kDynamic;
}

cudaError_t launch_bwd(const BwdParams& p, cudaStream_t stream) {
  if (p.d == 64)
    return p.fp16 ? launch_bwd_impl<64, true>(p, stream) : launch_bwd_impl<64, false>(p, stream);
  return p.fp16 ? launch_bwd_impl<128, true>(p, stream) : launch_bwd_impl<128, false>(p, stream);
}

cudaError_t read_and_clear_bwd_error(int* value) {
  cudaError_t err = cudaMemcpyFromSymbol(value, g_bwd_device_error, sizeof(int));
  if (err != cudaSuccess) return err;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_bwd_device_error, &zero, sizeof(int));
}

}  // namespace fa
