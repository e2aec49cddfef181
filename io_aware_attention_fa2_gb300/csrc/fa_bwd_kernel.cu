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
// Each step's dQ_i contribution is added to an fp32 workspace laid out [B, H, N, d] (one Q
// block's rows are one contiguous 128 x d block, which keeps the reductions' addresses
// compact); a pre-kernel computes D and clears the workspace, a post-kernel scales, rounds and
// transposes dQ back to [B, N, H, d].
//
// Per step (Q block i), all MMAs 128 x 128 x d or 128 x d x 128, fp32 accumulators in TMEM:
//   S^T  = K_j Q_i^T     (smem x smem)            -> T_S   lanes = keys, columns = queries
//   dP^T = V_j dO_i^T    (smem x smem)            -> T_dP
//   softmax warps: P^T = exp2(S^T scale log2e - LSE_i log2e) (masked), written back over T_S
//                  as 16-bit pairs and read back from there for dS^T = P^T (dP^T - D_i),
//                  stored as rows (queries contiguous, 128-byte swizzle) in shared memory.
//                  The factor scale of dS' = scale dS is applied to dK in its epilogue and
//                  to dQ when it is rounded.
//   dV  += P^T dO_i      (TMEM x smem, dO MN-major)
//   dQ_i^T = K_j^T dS^T  (smem x smem, both MN-major; d = 128)  -> T_dP, lanes = features
//   (d = 64: dQ_i = dS K_j, lanes = queries)
//   dK  += dS^T Q_i      (smem x smem: the same dS rows read K-major, Q MN-major)
//   dQ warps: dQ_i -> fp32 workspace (red.global.add: with lanes = features, one warp's
//             reduction for a query is one 128-byte line)
// MMA issue order: dV(i), then (after dS(i)) S^T(i+1), dQ(i), dK(i), then dP^T(i+1): keeping
// P^T(i) in TMEM until dS(i) has read it lets the softmax phases run as rolled loops (about a
// quarter of the code, no register copy of P^T); dQ(i)'s read-out overlaps dK(i), and the
// next dP^T waits only for that read-out.
// TMEM columns: T_S [0,128), T_dP [128,256), dV [256, 256+d), dK [256+d, 256+2d).
//
// Warps: 0 TMA producer (K_j, V_j once; Q_i, dO_i into a 2-deep ring), 1 MMA issuer and TMEM
// allocator, 2..5 softmax / dS (thread <-> TMEM lane), 6..9 dQ read-out and reduction.
// Every wait is bounded.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "ptx_sm103.cuh"

namespace fa {

// Error word of the backward kernels (the forward has its own): nonzero after a wait ran out.
__device__ int g_bwd_device_error = 0;

namespace {

// Warps: producer, MMA, 4 softmax / dS' warps (group 0), 4 dQ warps, and at d = 64 a second
// group of 4 softmax / dS' warps. With two groups, the two warps of a TMEM lane quarter share
// each key row: group g takes queries [64g, 64g + 64) of every step, which halves the length of
// the softmax and dS' phases each thread walks. At d = 64 those phases, not the products (half
// as long as at d = 128), set the step, and the second group gives their latencies twice the
// warps to hide behind.
template <int D>
struct BwdCfg {
  static constexpr int kSoftGroups = D == 64 ? 2 : 1;
  static constexpr int kThreads = 320 + 128 * (kSoftGroups - 1);
  // TMEM column of the packed P^T of 32-query chunk c (16 columns). Each group writes P over
  // the S^T columns it has itself read (a group must not overwrite columns another group may
  // still be loading): one group packs chunks 0..3 into columns 0..63 in order; two groups put
  // chunks 0, 1 in columns 0..31 and chunks 2, 3 in columns 64..95.
  static __host__ __device__ constexpr uint32_t p_col(int c) {
    return kSoftGroups == 2 ? (c / 2) * 64 + (c % 2) * 16 : c * 16;
  }
  // d = 64 leaves TMEM columns free, so P^T gets columns of its own [kT_P, kT_P + 64) instead of
  // sharing S^T's: then S^T(i+1) can be issued as soon as P^T(i) is written (with dV(i)), not
  // only after dS(i) has read P^T(i) back, and the next step's P phase need not wait for it.
  static constexpr bool kSeparateP = D == 64;
  static constexpr uint32_t kT_P = 256 + 2 * D;
  // TMEM column of P^T chunk c, from the allocation's base
  static __host__ __device__ constexpr uint32_t p_at(int c) {
    return kSeparateP ? kT_P + c * 16 : p_col(c);   // (kT_S = 0)
  }
  static_assert(!kSeparateP || kT_P + 64 <= 512, "TMEM columns");
};
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
  BB_DS_FULL,                              // dS^T rows in shared memory (128 arrivals)
  BB_DQ_FULL,                              // dQ_i (d = 128: dQ_i^T) in TMEM (T_dP)
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

// Four consecutive 16-bit elements (8 bytes) as fp32.
template <bool FP16>
__device__ __forceinline__ float4 load4(const void* p, int64_t i) {
  const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p) + i);
  float4 f;
  unpack2<FP16>(w.x, f.x, f.y);
  unpack2<FP16>(w.y, f.z, f.w);
  return f;
}

// D[b, h, q] = <dO[b, q, h, :], O[b, q, h, :]> and dQ workspace rows cleared. One warp per
// (b, q, h) row of the [B, N, H, d] tensors, 4 elements per lane.
template <int D, bool FP16>
__global__ void __launch_bounds__(256)
    fa_bwd_pre_kernel(const void* __restrict__ o, const void* __restrict__ dout,
                      float* __restrict__ dpre, float* __restrict__ dq_acc, int H, int N,
                      long long rows) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32;
  if (row >= rows) return;
  const int lane = threadIdx.x % 32;
  float acc = 0.f;
  if (4 * lane < D) {
    const float4 a = load4<FP16>(o, row * D + 4 * lane);
    const float4 g = load4<FP16>(dout, row * D + 4 * lane);
    acc = fmaf(a.x, g.x, fmaf(a.y, g.y, fmaf(a.z, g.z, a.w * g.w)));
    reinterpret_cast<float4*>(dq_acc + row * D)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    const long long h = row % H, bq = row / H;   // row = (b * N + q) * H + h
    const long long q = bq % N, b = bq / N;
    dpre[(b * H + h) * N + q] = acc;
  }
}

// Waits until the kernels this grid depends on (launched before it on the stream with
// programmatic stream serialisation) have completed and their writes are visible; returns at
// once when there is no such dependency.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// dQ[b, q, h, :] (input type) = scale x the workspace row [b, h, q, :] (which holds
// sum_j dS_qj k_j). One warp per (b, q, h) row, 4 elements per lane.
template <int D, bool FP16>
__global__ void __launch_bounds__(256)
    fa_bwd_post_kernel(const float* __restrict__ dq_acc, void* __restrict__ dq, float scale,
                       int H, int N, long long rows) {
  grid_dependency_wait();   // the main kernel's dQ partial sums
  const long long row = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32;
  if (row >= rows) return;
  const int lane = threadIdx.x % 32;
  if (4 * lane >= D) return;
  const long long h = row % H, bq = row / H;   // row = (b * N + q) * H + h
  const long long q = bq % N, b = bq / N;
  const float4 v = reinterpret_cast<const float4*>(dq_acc + ((b * H + h) * N + q) * D)[lane];
  reinterpret_cast<uint2*>(static_cast<uint16_t*>(dq) + row * D)[lane] =
      make_uint2(pack2<FP16>(v.x * scale, v.y * scale), pack2<FP16>(v.z * scale, v.w * scale));
}

// ---------------------------------------------------------------------------------------------
// P^T for 32 queries of this thread's key, packed to 16-bit pairs: 2^(S^T scale log2e -
// LSE log2e). l2 holds the 32 queries' LSE log2e (+inf for rows to ignore). MASKED: only the
// queries t of the chunk with lo <= t <= hi see the key (causal diagonal, window, keys past N or
// past the batch's key length).
template <bool MASKED, bool FP16>
__device__ __forceinline__ void p_chunk(const uint32_t (&sr)[32], const float* __restrict__ l2,
                                        float scale_log2, int lo, int hi,
                                        uint32_t* __restrict__ out) {
#pragma unroll
  for (int t4 = 0; t4 < 8; ++t4) {
    const float4 l = reinterpret_cast<const float4*>(l2)[t4];
    float x0, x1, x2, x3;
    ptx::fma2(x0, x1, __uint_as_float(sr[4 * t4]), __uint_as_float(sr[4 * t4 + 1]), scale_log2,
              scale_log2, -l.x, -l.y);
    ptx::fma2(x2, x3, __uint_as_float(sr[4 * t4 + 2]), __uint_as_float(sr[4 * t4 + 3]),
              scale_log2, scale_log2, -l.z, -l.w);
    if constexpr (MASKED) {
      if (4 * t4 < lo || 4 * t4 > hi) x0 = -INFINITY;
      if (4 * t4 + 1 < lo || 4 * t4 + 1 > hi) x1 = -INFINITY;
      if (4 * t4 + 2 < lo || 4 * t4 + 2 > hi) x2 = -INFINITY;
      if (4 * t4 + 3 < lo || 4 * t4 + 3 > hi) x3 = -INFINITY;
    }
    out[2 * t4] = pack2<FP16>(ptx::exp2_approx(x0), ptx::exp2_approx(x1));
    out[2 * t4 + 1] = pack2<FP16>(ptx::exp2_approx(x2), ptx::exp2_approx(x3));
  }
}

// dS^T = P^T (dP^T - D) for 32 queries, packed to 16-bit pairs (scale is applied to dQ, dK).
template <bool FP16>
__device__ __forceinline__ void ds_chunk(const uint32_t (&dr)[32], const uint32_t* __restrict__ pp,
                                         const float* __restrict__ dd, uint32_t (&out)[16]) {
#pragma unroll
  for (int t4 = 0; t4 < 8; ++t4) {
    const float4 dv = reinterpret_cast<const float4*>(dd)[t4];
    float p0, p1, p2, p3, e0, e1, e2, e3;
    unpack2<FP16>(pp[2 * t4], p0, p1);
    unpack2<FP16>(pp[2 * t4 + 1], p2, p3);
    ptx::add2(e0, e1, __uint_as_float(dr[4 * t4]), __uint_as_float(dr[4 * t4 + 1]), -dv.x,
              -dv.y);
    ptx::add2(e2, e3, __uint_as_float(dr[4 * t4 + 2]), __uint_as_float(dr[4 * t4 + 3]), -dv.z,
              -dv.w);
    ptx::mul2(e0, e1, e0, e1, p0, p1);
    ptx::mul2(e2, e3, e2, e3, p2, p3);
    out[2 * t4] = pack2<FP16>(e0, e1);
    out[2 * t4 + 1] = pack2<FP16>(e2, e3);
  }
}

template <int D, bool FP16>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_do, const float* __restrict__ lse,
                  const float* __restrict__ dpre, float* __restrict__ dq_acc,
                  void* __restrict__ dk_ptr, void* __restrict__ dv_ptr, int H, int N, int causal,
                  int window_left, int window_right, const int* __restrict__ seqlens_k,
                  float scale, float scale_log2, int heads_per_group) {
  using L = BwdSmem<D>;
  static_assert(L::kDynamic <= 227 * 1024, "backward tiles exceed shared memory");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  const uint32_t smem_base = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* const smem_gen = smem_raw + (smem_base - ptx::smem_addr(smem_raw));
  const uint32_t sK = smem_base + L::kK, sV = smem_base + L::kV;
  const uint32_t sQ = smem_base + L::kQ, sdO = smem_base + L::kdO, sdS = smem_base + L::kdS;
  float* const stat = reinterpret_cast<float*>(smem_gen + L::kStat);   // [2][128]
  auto bar = [&](int i) { return smem_base + L::kBars + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Unit: (b, h) x K/V block. Heads go in groups of `heads_per_group` (sized on the host so
  // that a group's Q, dO and dQ partial sums stay in L2); within a group, units go K/V block by
  // K/V block across the group's heads, longest (causal) walk first, so that the long walks of
  // the last group do not start at the end of the grid.
  const int num_kv = (N + BLOCK_N - 1) / BLOCK_N;
  const int num_q = (N + BLOCK_M - 1) / BLOCK_M;
  const int num_bh = static_cast<int>(gridDim.x) / num_kv;
  const int group_units = heads_per_group * num_kv;
  const int grp = static_cast<int>(blockIdx.x) / group_units;
  const int rem = static_cast<int>(blockIdx.x) % group_units;
  const int g_size = min(heads_per_group, num_bh - grp * heads_per_group);
  const int bh = grp * heads_per_group + rem % g_size;
  const int jb = rem / g_size;                              // K/V block (block 0 sees most Q)
  const int b = bh / H, h = bh % H;
  // Q blocks [i0, i0 + steps) hold a query that sees a key of this block: key j is visible to
  // query i when j < the batch's key length, j <= i (causal), j >= i - window_left and
  // j <= i + window_right (negative: no bound). Window bounds arrive clamped to [-1, N].
  const int len = seqlens_k ? min(max(seqlens_k[b], 0), N) : N;
  const int k0 = jb * BLOCK_N;
  int i0 = causal ? k0 / BLOCK_M : 0;
  if (window_right >= 0) i0 = max(i0, max(k0 - window_right, 0) / BLOCK_M);
  int i_end = num_q;
  if (window_left >= 0) i_end = min(i_end, (k0 + BLOCK_N - 1 + window_left) / BLOCK_M + 1);
  if (k0 >= len) i_end = i0;
  const int steps = max(i_end - i0, 0);
  if (steps == 0) {
    // No query sees a key of this block: dK = dV = 0 for its keys, nothing else to do.
    if (warp >= 2 && warp < 6) {
      const int key = k0 + (warp & 3) * 32 + lane;
      if (key < N) {
        for (int which = 0; which < 2; ++which) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(which ? dk_ptr : dv_ptr) +
                                                ((static_cast<int64_t>(b) * N + key) * H + h) * D);
#pragma unroll
          for (int t = 0; t < D / 8; ++t) dst[t] = make_uint4(0, 0, 0, 0);
        }
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(bar(BB_KV_FULL), 1);
    for (int s = 0; s < kBwdStages; ++s) {
      ptx::mbar_init(bar(BB_QD_FULL + s), 1);
      ptx::mbar_init(bar(BB_QD_EMPTY + s), 1);
    }
    ptx::mbar_init(bar(BB_S_FULL), 1);
    ptx::mbar_init(bar(BB_DP_FULL), 1);
    ptx::mbar_init(bar(BB_P_FULL), 128 * BwdCfg<D>::kSoftGroups);
    ptx::mbar_init(bar(BB_DS_FULL), 128 * BwdCfg<D>::kSoftGroups);
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
  // The softmax and dQ warps go on to warp-collective TMEM loads and stores after their waits.
  // They reach every wait converged, so their lanes read the barrier word, the abort flag and
  // the timer in the same instructions and leave it together; a per-warp vote (measured 3 %
  // slower here) is not needed.
  auto wait_w = [&](int slot, uint32_t parity) {
    return ptx::wait_bounded(bar(slot), parity, abort_p, kWaitLimitNs);
  };
  // D and the cleared dQ workspace come from the pre kernel, which may still be finishing:
  // the warps that read or reduce into them wait for it (the loads of K, V, Q, dO go ahead).
  if (warp >= 2) grid_dependency_wait();

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
      constexpr uint32_t id_st = ptx::idesc_f16(FP16, 128, BLOCK_M, false);   // S^T, dP^T
      constexpr uint32_t id_acc = ptx::idesc_f16(FP16, 128, D, true);         // dV, dK
      // d = 128: dQ^T = K_j^T dS'^T (M = features); d = 64: dQ = dS' K_j (M = queries).
      constexpr uint32_t id_dq = D == 128 ? ptx::idesc_f16(FP16, D, BLOCK_M, true, true)
                                          : ptx::idesc_f16(FP16, BLOCK_M, D, true, true);
      auto qbase = [&](int n) { return sQ + (n % kBwdStages) * L::kTile; };
      auto dobase = [&](int n) { return sdO + (n % kBwdStages) * L::kTile; };
      // Descriptors of the operands' bases: K-major (LBO 16) and MN-major (LBO = next box).
      const ptx::SmemDesc k_kmaj = ptx::smem_desc_sw128_split(sK, 16, 1024);
      const ptx::SmemDesc v_kmaj = ptx::smem_desc_sw128_split(sV, 16, 1024);
      const ptx::SmemDesc k_mn = ptx::smem_desc_sw128_split(sK, kBoxBytes, 1024);
      const ptx::SmemDesc ds_mn = ptx::smem_desc_sw128_split(sdS, kBoxBytes, 1024);
      const ptx::SmemDesc ds_kmaj = ptx::smem_desc_sw128_split(sdS, 16, 1024);
      // S^T = K_j Q_i^T -> T_S and dP^T = V_j dO_i^T -> T_dP: both operands K-major over d.
      auto issue_s = [&](int n) {
        ptx::tc_fence_after_sync();
        const ptx::SmemDesc q_desc = ptx::smem_desc_sw128_split(qbase(n), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * kBoxBytes + (kk % 4) * 32;
          ptx::mma_f16_ss(tmem + kT_S, k_kmaj.at(off), q_desc.at(off), id_st, kk > 0);
        }
        ptx::mma_commit(bar(BB_S_FULL));
      };
      auto issue_dp = [&](int n) {
        ptx::tc_fence_after_sync();
        const ptx::SmemDesc do_desc = ptx::smem_desc_sw128_split(dobase(n), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * kBoxBytes + (kk % 4) * 32;
          ptx::mma_f16_ss(tmem + kT_dP, v_kmaj.at(off), do_desc.at(off), id_st, kk > 0);
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
        const ptx::SmemDesc do_mn = ptx::smem_desc_sw128_split(dobase(n), kBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < BLOCK_M / 16; ++kk)
          ptx::mma_f16_ts(tmem + kT_dV, tmem + BwdCfg<D>::p_at(kk / 2) + (kk % 2) * 8,
                          do_mn.at(kk * 16 * 128), id_acc, (n > 0 || kk > 0) ? 1u : 0u);
        if constexpr (BwdCfg<D>::kSeparateP) {
          // S^T(i+1) right away: the softmax warps have read S^T(i) (P^T(i) is written), and
          // P^T(i) lives in columns of its own. P^T(i+1) is written only after S^T(i+1) has
          // completed, and so has dV(i), issued before it (in-order pipe).
          if (next) {
            if (!wait(BB_QD_FULL + (n + 1) % kBwdStages, ((n + 1) / kBwdStages) & 1)) {
              ok = false;
              break;
            }
            issue_s(n + 1);
          }
        }
        if (!wait(BB_DS_FULL, n & 1)) { ok = false; break; }
        if constexpr (!BwdCfg<D>::kSeparateP) {
          // S^T(i+1) over P^T(i): the softmax warps have read P^T(i) back for dS(i), and
          // dV(i), issued before, reads it first (in-order pipe).
          if (next) {
            if (!wait(BB_QD_FULL + (n + 1) % kBwdStages, ((n + 1) / kBwdStages) & 1)) {
              ok = false;
              break;
            }
            issue_s(n + 1);
          }
        }
        ptx::tc_fence_after_sync();
        // dQ first, into T_dP (dP^T(i) is in the softmax threads' registers by now), so that
        // its read-out overlaps dK. Both operands MN-major, 16 keys = 16 rows of 128 bytes per
        // MMA: the dS' rows (queries contiguous) and K_j (d contiguous).
#pragma unroll
        for (int kk = 0; kk < BLOCK_N / 16; ++kk) {
          const uint64_t ds_desc = ds_mn.at(kk * 16 * 128);
          const uint64_t k_desc = k_mn.at(kk * 16 * 128);
          if constexpr (D == 128)
            ptx::mma_f16_ss(tmem + kT_dP, k_desc, ds_desc, id_dq, kk > 0);
          else
            ptx::mma_f16_ss(tmem + kT_dP, ds_desc, k_desc, id_dq, kk > 0);
        }
        ptx::mma_commit(bar(BB_DQ_FULL));
        // dK += dS'^T Q_i: A = the same dS' rows read K-major (queries are the K dimension),
        // B = Q_i MN-major.
        const ptx::SmemDesc q_mn = ptx::smem_desc_sw128_split(qbase(n), kBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < BLOCK_M / 16; ++kk)
          ptx::mma_f16_ss(tmem + kT_dV + D, ds_kmaj.at((kk / 4) * kBoxBytes + (kk % 4) * 32),
                          q_mn.at(kk * 16 * 128), id_acc, (n > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(bar(BB_QD_EMPTY + s));   // Q_i and dO_i are no longer read
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
  } else if (warp < 6 || warp >= 10) {
    // ---------------------------------------------------------------- softmax / dS' warps
    // TMEM lane r = key jb * 128 + r for S^T, dP^T, dV, dK. Group g (warps 2..5: 0, 10..13: 1)
    // takes the 32-query chunks [c_beg, c_end) of every step and the 32-column chunks
    // [e_beg, e_end) of the dK, dV rows.
    constexpr int kGroups = BwdCfg<D>::kSoftGroups;
    const int grp_sm = warp >= 10 ? 1 : 0;
    const int c_beg = grp_sm * (BLOCK_M / 32 / kGroups), c_end = c_beg + BLOCK_M / 32 / kGroups;
    const int e_beg = grp_sm * (D / 32 / kGroups), e_end = e_beg + D / 32 / kGroups;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int key = jb * BLOCK_N + r;
    const bool key_ok = key < len;   // keys past N or past the batch's key length see no query
    // queries [q_lo, q_hi] see this key
    int q_lo = causal ? key : 0, q_hi = N - 1;
    if (window_right >= 0) q_lo = max(q_lo, key - window_right);
    if (window_left >= 0) q_hi = min(q_hi, key + window_left);
    uint8_t* const ds_gen = smem_gen + L::kdS;
    float* const s_lse = stat;         // LSE_i * log2e, +inf for rows to ignore
    float* const s_d = stat + 128;     // D_i
    bool ok = true;
    // Row statistics, one query per thread, fetched a step ahead. Queries past N (and rows
    // with no allowed key, LSE = -inf) get +inf, so their P is 0.
    float l2_next = INFINITY, d_next = 0.f;
    auto fetch_stats = [&](int n) {
      const int q = (i0 + n) * BLOCK_M + r;
      l2_next = INFINITY;
      d_next = 0.f;
      if (q < N) {
        const float lv = lse[static_cast<int64_t>(bh) * N + q];
        if (lv != -INFINITY) l2_next = lv * kLog2e;
        d_next = dpre[static_cast<int64_t>(bh) * N + q];
      }
    };
    // Group 0 fetches and stages the statistics; every group reads them.
    if (grp_sm == 0) fetch_stats(0);
    for (int n = 0; n < steps; ++n) {
      const int q0 = (i0 + n) * BLOCK_M;
      // One buffer serves every step: it is refilled only after every softmax thread has
      // finished the previous step's dS' (DS_FULL), the last phase that reads it.
      if (n > 0 && !wait_w(BB_DS_FULL, (n - 1) & 1)) { ok = false; break; }
      if (grp_sm == 0) {
        s_lse[r] = l2_next;
        s_d[r] = d_next;
        ptx::mbar_arrive(bar(BB_STAT));
      }
      if (!wait_w(BB_STAT, n & 1)) { ok = false; break; }
      if (grp_sm == 0 && n + 1 < steps) fetch_stats(n + 1);

      // --- P^T: this thread's key against the 128 queries of block i, kept packed as 16-bit
      // pairs (the values the dV product uses, also used for dS'). Query q0 + t sees the key
      // only if key <= q0 + t (causal); keys past N do not exist.
      if (!wait_w(BB_S_FULL, n & 1)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      // this step's query range of the key, relative to the block (empty when !key_ok)
      const int lo = key_ok ? q_lo - q0 : BLOCK_M, hi = key_ok ? q_hi - q0 : -1;
      // P^T stays in TMEM (over S^T columns this group has read, BwdCfg::p_col) until dS(i)
      // has read it back.
#pragma unroll 1
      for (int c = c_beg; c < c_end; ++c) {
        uint32_t sr[32];
        ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_S + c * 32, sr);
        ptx::tmem_wait_ld();
        ptx::reg_fence(sr);
        uint32_t pr[16];
        if (lo > 32 * c || hi < 32 * c + 31)
          p_chunk<true, FP16>(sr, s_lse + 32 * c, scale_log2, lo - 32 * c, hi - 32 * c, pr);
        else
          p_chunk<false, FP16>(sr, s_lse + 32 * c, scale_log2, 0, 31, pr);
        ptx::tmem_st_32x32b_x16(tmem + lane_off + BwdCfg<D>::p_at(c), pr);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before_sync();
      ptx::mbar_arrive(bar(BB_P_FULL));

      // --- dS^T = P^T (dP^T - D) -> rows of dS^T (queries contiguous) in shared memory, which
      // both the dQ and the dK products read. dP^T(i) was issued after dQ(i-1) and dK(i-1)
      // completed, so the buffer is free again.
      if (!wait_w(BB_DP_FULL, n & 1)) { ok = false; break; }
      ptx::tc_fence_after_sync();
#pragma unroll 1
      for (int c = c_beg; c < c_end; ++c) {
        uint32_t dr[32], pw[16];
        ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_dP + c * 32, dr);
        ptx::tmem_ld_32x32b_x16(tmem + lane_off + BwdCfg<D>::p_at(c), pw);
        ptx::tmem_wait_ld();
        ptx::reg_fence(dr);
        ptx::reg_fence(pw);
        uint32_t pk[16];
        ds_chunk<FP16>(dr, pw, s_d + 32 * c, pk);
        // queries 32c .. 32c+31 of key row r: 4 chunks of 16 bytes in box c / 2, swizzled
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = (c % 2) * 4 + u;        // 16-byte chunk within the 128-byte row
          const uint32_t off = (c / 2) * kBoxBytes + r * 128 + ((chunk ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(ds_gen + off) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before_sync();
      ptx::mbar_arrive(bar(BB_DS_FULL));
    }
    // dK (times scale), dV rows once every MMA of this CTA has completed.
    if (ok && !wait_w(BB_MMA_DONE, 0)) ok = false;
    if (ok) {
      ptx::tc_fence_after_sync();
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        uint16_t* out = static_cast<uint16_t*>(which ? dk_ptr : dv_ptr) +
                        ((static_cast<int64_t>(b) * N + key) * H + h) * D;
        const float f = which ? scale : 1.f;
#pragma unroll 1
        for (int c = e_beg; c < e_end; ++c) {
          uint32_t gr[32];
          ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_dV + which * D + c * 32, gr);
          ptx::tmem_wait_ld();
          ptx::reg_fence(gr);
          if (key < N) {
            uint4* dst = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              float g[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) g[e] = __uint_as_float(gr[8 * t + e]) * f;
              dst[t] = make_uint4(pack2<FP16>(g[0], g[1]), pack2<FP16>(g[2], g[3]),
                                  pack2<FP16>(g[4], g[5]), pack2<FP16>(g[6], g[7]));
            }
          }
        }
      }
    } else {
      record_timeout(abort_p);
    }
  } else {
    // ---------------------------------------------------------------- dQ warps
    // The whole dQ block is loaded out of TMEM before T_dP is released, then reduced into the
    // fp32 workspace. d = 128: TMEM lane = feature, column = query, so one warp's reduction
    // for a query covers 32 consecutive features (one 128-byte line). d = 64: lane = query.
    const int quarter = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    for (int n = 0; n < steps; ++n) {
      const int q0 = (i0 + n) * BLOCK_M;
      if (!wait_w(BB_DQ_FULL, n & 1)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      if constexpr (D == 128) {
        uint32_t v0[32], v1[32], v2[32], v3[32];
        ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_dP + 0, v0);
        ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_dP + 32, v1);
        ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_dP + 64, v2);
        ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_dP + 96, v3);
        ptx::tmem_wait_ld();
        ptx::reg_fence(v0);
        ptx::reg_fence(v1);
        ptx::reg_fence(v2);
        ptx::reg_fence(v3);
        ptx::tc_fence_before_sync();
        ptx::mbar_arrive(bar(BB_DQ_TAKEN));
        const int nq = min(BLOCK_M, N - q0);
        const int64_t stride = D;
        float* const base =
            dq_acc + (static_cast<int64_t>(bh) * N + q0) * D + quarter * 32 + lane;
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (t < nq) ptx::red_add_f32(base + t * stride, __uint_as_float(v0[t]));
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (32 + t < nq) ptx::red_add_f32(base + (32 + t) * stride, __uint_as_float(v1[t]));
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (64 + t < nq) ptx::red_add_f32(base + (64 + t) * stride, __uint_as_float(v2[t]));
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (96 + t < nq) ptx::red_add_f32(base + (96 + t) * stride, __uint_as_float(v3[t]));
      } else {
        uint32_t v0[32], v1[32];
        ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_dP + 0, v0);
        ptx::tmem_ld_32x32b_x32(tmem + lane_off + kT_dP + 32, v1);
        ptx::tmem_wait_ld();
        ptx::reg_fence(v0);
        ptx::reg_fence(v1);
        ptx::tc_fence_before_sync();
        ptx::mbar_arrive(bar(BB_DQ_TAKEN));
        const int r = quarter * 32 + lane;
        if (q0 + r < N) {
          float* dst = dq_acc + (static_cast<int64_t>(bh) * N + q0 + r) * D;
#pragma unroll
          for (int t = 0; t < 32; t += 4)
            ptx::red_add_v4(dst + t, __uint_as_float(v0[t]), __uint_as_float(v0[t + 1]),
                            __uint_as_float(v0[t + 2]), __uint_as_float(v0[t + 3]));
#pragma unroll
          for (int t = 0; t < 32; t += 4)
            ptx::red_add_v4(dst + 32 + t, __uint_as_float(v1[t]), __uint_as_float(v1[t + 1]),
                            __uint_as_float(v1[t + 2]), __uint_as_float(v1[t + 3]));
        }
      }
    }
    if (!ok) record_timeout(abort_p);
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
  const long long bh = static_cast<long long>(p.B) * p.H;
  // Heads per dispatch group: the group's Q and dO (2 bytes each) and dQ partial sums (4 bytes)
  // within ~64 MiB of L2.
  const long long bytes_per_head = 8ll * p.N * p.d;
  const int heads_per_group =
      static_cast<int>(std::max(1ll, std::min(bh, (64ll << 20) / bytes_per_head)));
  // The main and post kernels are launched with programmatic stream serialisation: each may
  // start (set-up, independent loads) while the kernel before it finishes, and waits for it
  // in the kernel before touching what it wrote.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_kv * bh));
  cfg.blockDim = dim3(BwdCfg<D>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kernel, p.tm_q, p.tm_k, p.tm_v, p.tm_do, p.lse,
                           static_cast<const float*>(p.dpre), p.dq_acc, p.dk, p.dv, p.H, p.N,
                           p.causal, p.window_left, p.window_right, p.seqlens_k, p.scale,
                           p.scale * kLog2e, heads_per_group);
  if (err != cudaSuccess) return err;
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, fa_bwd_post_kernel<D, FP16>,
                            static_cast<const float*>(p.dq_acc), p.dq, p.scale, p.H, p.N, rows);
}

}  // namespace

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
