// fa_fwd_kernel.cu -- fused attention forward for sm_103a: TMA + tcgen05/TMEM + online softmax.
//
// What one CTA computes ("FlashAttention 优化原理与实现要点解析" §5, with the loop order of §7
// and "FlashAttention V2 核心原理与架构设计" §2.2 V2: Q blocks outside, K/V blocks inside):
//
//   for its unit (b, h, Q tile i of 128 rows):
//     load Q_i once
//     for each K/V tile j (j <= i when causal; tiles above the diagonal are skipped, §7):
//       S = Q_i K_j^T                          (tcgen05.mma, fp32 accumulator in TMEM)
//       mask: key > query (causal), key >= N (ragged tail)
//       m_new = max(m, rowmax(S) * scale)      (online softmax, §4.2; log2 units here)
//       P = exp(S * scale - m_new); alpha = exp(m - m_new)
//       l = alpha * l + rowsum(P)
//       O = alpha * O + P V_j                  (§4.3; O rescaled in TMEM, P V by tcgen05.mma)
//     O /= l once at the end (§6: numerator and denominator kept apart), LSE = m + ln l
//
// Work split inside the CTA (the Blackwell form of the split-Q partition of
// "FlashAttention v1 & v2 笔记" §五.3: every row belongs to exactly one thread, so row
// statistics never need a cross-warp reduction):
//   warp 0        TMA producer: Q once, then K_j / V_j into a STAGES-deep shared-memory ring
//   warp 1        TMEM allocator + MMA issuer (one thread): S_j into one of two TMEM S buffers,
//                 O += P_j V_j into the TMEM O accumulator
//   warps 2..5    softmax: thread <-> query row (TMEM lane); reads S_j from TMEM, writes P_j
//                 (rounded to the input type) into shared memory in the MMA operand layout,
//                 rescales O in TMEM, and finally normalises and stores O and LSE.
//
// TMEM columns: S buffer 0 at [0,128), S buffer 1 at [128,256), O at [256, 256+d).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "ptx_sm103.cuh"

namespace fa {

// Device error word: nonzero after a kernel wait ran past its limit. Read and cleared by
// read_and_clear_device_error.
__device__ int g_device_error = 0;

namespace {

constexpr int kStages = 2;                     // K/V ring depth
constexpr int kThreads = 192;                  // 6 warps
constexpr uint32_t kBoxBytes = BOX_ROWS * BOX_COLS * 2;   // 16 KiB
constexpr uint32_t kPBytes = 2 * kBoxBytes;               // 128 x 128 16-bit
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS0 = 0, kTmemO = 256;
constexpr uint64_t kWaitLimitNs = 1000000000ull;          // 1 s per wait
constexpr int kErrTimeout = -8;                            // FA_ERR_TIMEOUT

template <int D>
struct SmemLayout {
  static constexpr uint32_t kTile = (D / BOX_COLS) * kBoxBytes;    // Q, K or V tile
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kTile;
  static constexpr uint32_t kV = kK + kStages * kTile;
  static constexpr uint32_t kP = kV + kStages * kTile;
  static constexpr uint32_t kBars = kP + kPBytes;
  static constexpr uint32_t kNumBars = 16;
  static constexpr uint32_t kEnd = kBars + kNumBars * 8;
  static constexpr uint32_t kDynamic = kEnd + 1024;                // slack for 1 KiB alignment
};

// Barrier slots.
enum : int {
  BAR_Q_FULL = 0,
  BAR_K_FULL = 1,                    // + stage
  BAR_V_FULL = BAR_K_FULL + kStages,  // + stage
  BAR_KV_EMPTY = BAR_V_FULL + kStages,
  BAR_S_FULL = BAR_KV_EMPTY + kStages,  // + buffer (2)
  BAR_P_FULL = BAR_S_FULL + 2,
  BAR_O_READY = BAR_P_FULL + 1,
  BAR_MMA_DONE = BAR_O_READY + 1,
  BAR_COUNT = BAR_MMA_DONE + 1
};
static_assert(BAR_COUNT <= 16, "barrier slots");

__device__ __forceinline__ void record_timeout(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(&g_device_error, 0, kErrTimeout);
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

// ---------------------------------------------------------------------------------------------
template <int D, bool FP16>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, void* __restrict__ o_ptr,
                  float* __restrict__ lse_ptr, int H, int N, int causal, float scale_log2) {
  using L = SmemLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  const uint32_t smem_base = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = smem_base + L::kQ;
  const uint32_t sK = smem_base + L::kK;
  const uint32_t sV = smem_base + L::kV;
  const uint32_t sP = smem_base + L::kP;
  uint8_t* const sP_ptr = smem_raw + (sP - ptx::smem_addr(smem_raw));
  auto bar = [&](int i) { return smem_base + L::kBars + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // Work unit: (b, h) from blockIdx.x, Q tile from blockIdx.y. Causal units are dispatched
  // longest first (the last Q tile has the most K/V tiles).
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh % H;
  const int num_q_tiles = gridDim.y;
  const int q_tile = causal ? (num_q_tiles - 1 - static_cast<int>(blockIdx.y))
                            : static_cast<int>(blockIdx.y);
  const int num_kv_total = (N + BLOCK_N - 1) / BLOCK_N;
  const int num_kv = causal ? min(q_tile + 1, num_kv_total) : num_kv_total;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(bar(BAR_Q_FULL), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(BAR_K_FULL + s), 1);
      ptx::mbar_init(bar(BAR_V_FULL + s), 1);
      ptx::mbar_init(bar(BAR_KV_EMPTY + s), 1);
    }
    ptx::mbar_init(bar(BAR_S_FULL + 0), 1);
    ptx::mbar_init(bar(BAR_S_FULL + 1), 1);
    ptx::mbar_init(bar(BAR_P_FULL), 128);
    ptx::mbar_init(bar(BAR_O_READY), 1);
    ptx::mbar_init(bar(BAR_MMA_DONE), 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tm_q);
      ptx::prefetch_tensormap(&tm_k);
      ptx::prefetch_tensormap(&tm_v);
      const int q_row0 = q_tile * BLOCK_M;
      ptx::mbar_arrive_expect_tx(bar(BAR_Q_FULL), L::kTile);
      for (int c = 0; c < D / BOX_COLS; ++c)
        ptx::tma_load_4d(sQ + c * kBoxBytes, &tm_q, bar(BAR_Q_FULL), c * BOX_COLS, h, q_row0, b);
      int issued = 0;
      for (int j = 0; j < num_kv; ++j) {
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        if (!ptx::wait_bounded(bar(BAR_KV_EMPTY + s), ph ^ 1, abort_p, kWaitLimitNs)) {
          record_timeout(abort_p);
          break;
        }
        const int kv_row0 = j * BLOCK_N;
        ptx::mbar_arrive_expect_tx(bar(BAR_K_FULL + s), L::kTile);
        for (int c = 0; c < D / BOX_COLS; ++c)
          ptx::tma_load_4d(sK + s * L::kTile + c * kBoxBytes, &tm_k, bar(BAR_K_FULL + s),
                           c * BOX_COLS, h, kv_row0, b);
        ptx::mbar_arrive_expect_tx(bar(BAR_V_FULL + s), L::kTile);
        for (int c = 0; c < D / BOX_COLS; ++c)
          ptx::tma_load_4d(sV + s * L::kTile + c * kBoxBytes, &tm_v, bar(BAR_V_FULL + s),
                           c * BOX_COLS, h, kv_row0, b);
        issued = j + 1;
      }
      // Do not leave the CTA with copies in flight: wait (bounded) for the last load of every
      // stage and for Q. On the normal path these phases completed long ago.
      ptx::wait_bounded(bar(BAR_Q_FULL), 0, abort_p, kWaitLimitNs);
      for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j) {
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        ptx::wait_bounded(bar(BAR_K_FULL + s), ph, abort_p, kWaitLimitNs);
        ptx::wait_bounded(bar(BAR_V_FULL + s), ph, abort_p, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = ptx::idesc_f16(FP16, BLOCK_M, BLOCK_N, false);
      constexpr uint32_t idesc_pv = ptx::idesc_f16(FP16, BLOCK_M, D, true);
      bool ok = ptx::wait_bounded(bar(BAR_Q_FULL), 0, abort_p, kWaitLimitNs);
      // S_jj = Q K_jj^T into S buffer jj % 2.
      auto issue_s = [&](int jj) -> bool {
        const int s = jj % kStages;
        if (!ptx::wait_bounded(bar(BAR_K_FULL + s), (jj / kStages) & 1, abort_p, kWaitLimitNs))
          return false;
        ptx::tc_fence_after_sync();
        const uint32_t d_tmem = tmem + kTmemS0 + (jj & 1) * BLOCK_N;
        const uint32_t k_base = sK + s * L::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // 16 elements (32 bytes) of d per MMA; 4 steps per 128-byte swizzle span, then the
          // next 64-column box.
          const uint32_t off = (kk / 4) * kBoxBytes + (kk % 4) * 32;
          ptx::mma_f16_ss(d_tmem, ptx::smem_desc_sw128(sQ + off, 16, 1024),
                          ptx::smem_desc_sw128(k_base + off, 16, 1024), idesc_qk, kk > 0);
        }
        ptx::mma_commit(bar(BAR_S_FULL + (jj & 1)));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < num_kv; ++j) {
        if (j + 1 < num_kv && !issue_s(j + 1)) { ok = false; break; }
        const int s = j % kStages;
        if (!ptx::wait_bounded(bar(BAR_P_FULL), j & 1, abort_p, kWaitLimitNs) ||
            !ptx::wait_bounded(bar(BAR_V_FULL + s), (j / kStages) & 1, abort_p, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after_sync();
        const uint32_t v_base = sV + s * L::kTile;
#pragma unroll
        for (int kk = 0; kk < BLOCK_N / 16; ++kk) {
          // A = P (K-major over keys, two 64-key boxes); B = V tile (MN-major: d contiguous),
          // 16 keys = 16 rows of 128 bytes per step; LBO = next 64-column box of V.
          const uint32_t a_off = (kk / 4) * kBoxBytes + (kk % 4) * 32;
          const uint32_t b_off = kk * 16 * 128;
          ptx::mma_f16_ss(tmem + kTmemO, ptx::smem_desc_sw128(sP + a_off, 16, 1024),
                          ptx::smem_desc_sw128(v_base + b_off, kBoxBytes, 1024), idesc_pv,
                          (j > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(bar(BAR_KV_EMPTY + s));
        ptx::mma_commit(bar(BAR_O_READY));
      }
      if (!ok) record_timeout(abort_p);
      // Every MMA this thread issued has completed before TMEM can be released.
      ptx::mma_commit(bar(BAR_MMA_DONE));
      ptx::wait_bounded(bar(BAR_MMA_DONE), 0, abort_p, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int quarter = warp & 3;                       // TMEM lanes [32q, 32q+32)
    const int row = quarter * 32 + lane;                // query row within the tile
    const int q_idx = q_tile * BLOCK_M + row;           // query position
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool scale_pos = scale_log2 > 0.f;
    float m = -INFINITY;   // running max of scaled scores, log2 units
    float l = 0.f;         // running sum of 2^(x - m)
    bool ok = true;

    for (int j = 0; j < num_kv; ++j) {
      if (!ptx::wait_bounded(bar(BAR_S_FULL + (j & 1)), (j >> 1) & 1, abort_p, kWaitLimitNs)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after_sync();
      uint32_t sr[BLOCK_N / 32][32];
#pragma unroll
      for (int c = 0; c < BLOCK_N / 32; ++c)
        ptx::tmem_ld_32x32b_x32(t_lane + kTmemS0 + (j & 1) * BLOCK_N + c * 32, sr[c]);
      ptx::tmem_wait_ld();
      float s[BLOCK_N];
#pragma unroll
      for (int c = 0; c < BLOCK_N / 32; ++c) {
        ptx::reg_fence(sr[c]);
#pragma unroll
        for (int x = 0; x < 32; ++x) s[c * 32 + x] = __uint_as_float(sr[c][x]);
      }

      const int k0 = j * BLOCK_N;
      const bool need_mask = (causal && k0 + BLOCK_N - 1 > q_tile * BLOCK_M) || (k0 + BLOCK_N > N);
      if (!scale_pos) {
#pragma unroll
        for (int t = 0; t < BLOCK_N; ++t) s[t] *= scale_log2;
      }
      if (need_mask) {
        const int lim = causal ? min(q_idx + 1, N) : N;   // keys [0, lim) are allowed
#pragma unroll
        for (int t = 0; t < BLOCK_N; ++t)
          if (k0 + t >= lim) s[t] = -INFINITY;
      }
      float mt = -INFINITY;
#pragma unroll
      for (int t = 0; t < BLOCK_N; ++t) mt = fmaxf(mt, s[t]);
      const float m_tile = scale_pos ? mt * scale_log2 : mt;
      const float m_new = fmaxf(m, m_tile);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ptx::exp2_approx(m - m_use);
      float rs = 0.f;
      if (scale_pos) {
#pragma unroll
        for (int t = 0; t < BLOCK_N; ++t) {
          const float p = ptx::exp2_approx(fmaf(s[t], scale_log2, -m_use));
          s[t] = p;
          rs += p;
        }
      } else {
#pragma unroll
        for (int t = 0; t < BLOCK_N; ++t) {
          const float p = ptx::exp2_approx(s[t] - m_use);
          s[t] = p;
          rs += p;
        }
      }
      l = l * alpha + rs;
      m = m_new;

      if (j > 0) {
        // P V_{j-1} must be complete before O is rescaled and before P_j overwrites P_{j-1}.
        if (!ptx::wait_bounded(bar(BAR_O_READY), (j - 1) & 1, abort_p, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after_sync();
        if (!__all_sync(0xffffffffu, alpha == 1.f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orr[32];
            ptx::tmem_ld_32x32b_x32(t_lane + kTmemO + c * 32, orr);
            ptx::tmem_wait_ld();
            ptx::reg_fence(orr);
#pragma unroll
            for (int x = 0; x < 32; ++x)
              orr[x] = __float_as_uint(__uint_as_float(orr[x]) * alpha);
            ptx::tmem_st_32x32b_x32(t_lane + kTmemO + c * 32, orr);
          }
          ptx::tmem_wait_st();
        }
      }

      // P_j -> shared memory, K-major with the 128-byte swizzle: row `row`, 16-byte chunk c
      // of each 64-key box lands at chunk position c ^ (row % 8).
#pragma unroll
      for (int c = 0; c < BLOCK_N / 8; ++c) {
        uint4 v;
        v.x = pack2<FP16>(s[8 * c + 0], s[8 * c + 1]);
        v.y = pack2<FP16>(s[8 * c + 2], s[8 * c + 3]);
        v.z = pack2<FP16>(s[8 * c + 4], s[8 * c + 5]);
        v.w = pack2<FP16>(s[8 * c + 6], s[8 * c + 7]);
        const uint32_t off = (c / 8) * kBoxBytes + row * 128 + (((c % 8) ^ (row & 7)) << 4);
        *reinterpret_cast<uint4*>(sP_ptr + off) = v;
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before_sync();
      ptx::mbar_arrive(bar(BAR_P_FULL));
    }

    // ---------------------------------------------------------------- epilogue
    if (ok && ptx::wait_bounded(bar(BAR_O_READY), (num_kv - 1) & 1, abort_p, kWaitLimitNs)) {
      ptx::tc_fence_after_sync();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool valid = q_idx < N;
      using elem_t = uint16_t;
      elem_t* out_row = static_cast<elem_t*>(o_ptr) +
                        ((static_cast<int64_t>(b) * N + q_idx) * H + h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orr[32];
        ptx::tmem_ld_32x32b_x32(t_lane + kTmemO + c * 32, orr);
        ptx::tmem_wait_ld();
        ptx::reg_fence(orr);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(out_row + c * 32);
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            uint4 v;
            v.x = pack2<FP16>(__uint_as_float(orr[8 * x + 0]) * inv_l,
                              __uint_as_float(orr[8 * x + 1]) * inv_l);
            v.y = pack2<FP16>(__uint_as_float(orr[8 * x + 2]) * inv_l,
                              __uint_as_float(orr[8 * x + 3]) * inv_l);
            v.z = pack2<FP16>(__uint_as_float(orr[8 * x + 4]) * inv_l,
                              __uint_as_float(orr[8 * x + 5]) * inv_l);
            v.w = pack2<FP16>(__uint_as_float(orr[8 * x + 6]) * inv_l,
                              __uint_as_float(orr[8 * x + 7]) * inv_l);
            dst[x] = v;
          }
        }
      }
      if (valid)
        lse_ptr[(static_cast<int64_t>(b) * H + h) * N + q_idx] =
            (m + __log2f(l)) * 0.69314718055994530942f;
    } else if (ok) {
      record_timeout(abort_p);
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
cudaError_t launch_impl(const FwdParams& p, cudaStream_t stream) {
  auto kernel = fa_fwd_kernel<D, FP16>;
  const size_t smem = SmemLayout<D>::kDynamic;
  // Attribute set on every call: cheap, and correct for whichever device is current.
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int num_q_tiles = (p.N + BLOCK_M - 1) / BLOCK_M;
  dim3 grid(p.B * p.H, num_q_tiles, 1);
  kernel<<<grid, kThreads, smem, stream>>>(p.tm_q, p.tm_k, p.tm_v, p.o, p.lse, p.H, p.N,
                                           p.causal, p.scale_log2);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_smem_bytes(int d) {
  return d == 64 ? SmemLayout<64>::kDynamic : SmemLayout<128>::kDynamic;
}

cudaError_t launch_fwd(const FwdParams& p, cudaStream_t stream) {
  if (p.d == 64) return p.fp16 ? launch_impl<64, true>(p, stream) : launch_impl<64, false>(p, stream);
  return p.fp16 ? launch_impl<128, true>(p, stream) : launch_impl<128, false>(p, stream);
}

cudaError_t read_and_clear_device_error(cudaStream_t stream, int* value) {
  cudaError_t err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return err;
  err = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
  if (err != cudaSuccess) return err;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace fa
