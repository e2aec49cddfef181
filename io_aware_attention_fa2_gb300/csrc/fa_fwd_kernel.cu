// fa_fwd_kernel.cu -- fused attention forward for sm_103a: TMA + tcgen05/TMEM + online softmax.
//
// What one CTA computes ("FlashAttention 优化原理与实现要点解析" §5, with the loop order of §7
// and "FlashAttention V2 核心原理与架构设计" §2.2 V2: Q blocks outside, K/V blocks inside):
//
//   for its unit (b, h, Q block of 256 rows = Q tiles A and B of 128 rows each):
//     load Q_A, Q_B once
//     for each K/V tile j of 128 keys (only tiles at or below the diagonal when causal; the
//     tiles above it are never loaded, §7):
//       for X in {A, B}:
//         S_X = Q_X K_j^T                       (tcgen05.mma, fp32 accumulator in TMEM)
//         mask: key > query (causal), key >= N (ragged tail)
//         m_new = max(m, rowmax(scale * S_X))   (online softmax, §4.2; log2 units here)
//         P_X = exp(scale * S_X - m_new); alpha = exp(m - m_new); l = alpha * l + rowsum(P_X)
//         O_X = alpha * O_X + P_X V_j           (§4.3)
//     O_X /= l once at the end (§6: numerator and denominator kept apart); LSE = m + ln l
//
// Work split inside the CTA. Every query row belongs to exactly one thread, so row statistics
// never need a cross-warp reduction (the split-Q partition of "FlashAttention v1 & v2 笔记"
// §五.3, in its Blackwell form: a TMEM lane is a row):
//   warp 0       TMA producer: Q_A and Q_B once, then K_j and V_j into two 2-deep rings
//   warp 1       TMEM allocator and MMA issuer (one thread)
//   warps 2..5   softmax of tile A; warps 6..9 softmax of tile B. Each thread reads its row of
//                S_X from TMEM, writes P_X back over the same columns as packed 16-bit values,
//                rescales its row of O_X in TMEM when needed, and at the end normalises and
//                stores O_X and LSE.
//
// P never leaves tensor memory: the P V product takes its A operand straight from TMEM. The
// tensor pipe executes one thread's MMAs in issue order, which gives the reuse rules below
// without extra waits:
//   * S_X(j+1) is issued after P_X(j) V_j, so it may overwrite the columns holding P_X(j);
//   * when S_X(j+1) completes, P_X(j) V_j has completed too, so the softmax warps may rescale
//     O_X as soon as they see S_X(j+1).
// Issue order: S_A(0) S_B(0) | PV_A(0) S_A(1) PV_B(0) S_B(1) | PV_A(1) S_A(2) ... so the tensor
// pipe works on one tile while the other tile's softmax runs.
//
// Lazy rescaling: a warp keeps the exponent offset m of its rows until some row's maximum
// exceeds it by more than kRescaleLog2 (2^8); then every row of the warp moves to its exact
// running maximum and O and l are rescaled. In between, P <= 2^8 and O, l share the same
// offset, so O / l and m + log2(l) are exact in real arithmetic.
//
// TMEM columns (512 allocated): S_A [0,128), S_B [128,256), O_A [256,256+d), O_B [256+d,256+2d).
//
// The one-tile CTA (d = 64 without split K/V; Cfg below) runs tile A alone with warps 2..5 and
// two CTAs per SM: TMEM (256 allocated) S [0,128), O [128,192), P [192,256). With P in columns
// of its own, S(j+1) is issued as soon as the softmax has loaded S(j), and the softmax waits for
// P(j-1) V_{j-1} before it writes P(j) or rescales O.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "fa_internal.h"
#include "ptx_sm103.cuh"

namespace fa {

// Device error word: nonzero after a kernel wait ran past its limit. Read and cleared by
// read_and_clear_device_error.
__device__ int g_device_error = 0;

namespace {

constexpr int kStages = 2;                     // depth of the K ring and of the V ring
constexpr int kMaxQTiles = 2;                  // 128-row Q tiles per CTA: 2, or 1 (see Cfg)
constexpr uint32_t kBoxBytes = BOX_ROWS * BOX_COLS * 2;   // 16 KiB
constexpr uint64_t kWaitLimitNs = 1000000000ull;          // 1 s per wait
constexpr int kErrTimeout = -8;                            // FA_ERR_TIMEOUT
constexpr float kRescaleLog2 = 8.0f;

// Shape of one CTA. QT = 2: two Q tiles (A, B) whose softmax phases alternate on the tensor
// pipe; 512 TMEM columns (S_A, S_B, O_A, O_B), one CTA per SM. QT = 1 (d = 64 only): one Q
// tile, S 128 + O 64 + P 64 columns in a 256-column allocation, 6 warps and 80 KiB of shared
// memory, so that two CTAs share an SM; with P in columns of its own, S(j+1) is computed while
// the softmax of S(j) runs and P(j) V_j while the softmax of S(j+1) runs.
template <int QT, int D>
struct Cfg {
  static constexpr int kThreads = 64 + 128 * QT;
  static constexpr int kMinBlocks = QT == 1 && D == 64 ? 2 : 1;
  static constexpr uint32_t kTmemO = 128 * QT;                     // O_X at kTmemO + x * D
  static constexpr uint32_t kTmemCols = QT == 1 && D == 64 ? 256 : 512;
  // QT = 1: P in columns of its own after O (S 128 + O 64 + P 64 = 256), so that S(j+1) can
  // be computed while the softmax of S(j) runs. QT = 2: P is written over S.
  static constexpr bool kSeparateP = QT == 1;
  static constexpr uint32_t kTmemP = kTmemO + QT * D;
  static_assert(kTmemO + QT * D + (kSeparateP ? 64 : 0) <= kTmemCols, "TMEM columns");
};

template <int QT, int D>
struct SmemLayout {
  static constexpr uint32_t kTile = (D / BOX_COLS) * kBoxBytes;    // one Q, K or V tile
  static constexpr uint32_t kQ = 0;                                 // Q_A (, Q_B)
  static constexpr uint32_t kK = kQ + QT * kTile;
  static constexpr uint32_t kV = kK + kStages * kTile;
  static constexpr uint32_t kBars = kV + kStages * kTile;
  static constexpr uint32_t kNumBars = 24;
  static constexpr uint32_t kEnd = kBars + kNumBars * 8;
  static constexpr uint32_t kDynamic = kEnd + 1024;                // slack for 1 KiB alignment
};

// Barrier slots.
enum : int {
  BAR_Q_FULL = 0,
  BAR_K_FULL = 1,                         // + stage
  BAR_K_EMPTY = BAR_K_FULL + kStages,     // + stage
  BAR_V_FULL = BAR_K_EMPTY + kStages,     // + stage
  BAR_V_EMPTY = BAR_V_FULL + kStages,     // + stage
  BAR_S_FULL = BAR_V_EMPTY + kStages,     // + tile: S_X(j) computed (and all earlier MMAs)
  BAR_P_FULL = BAR_S_FULL + kMaxQTiles,   // + tile: P_X(j) in TMEM, O_X rescaled (128 arrivals)
  BAR_O_DONE = BAR_P_FULL + kMaxQTiles,   // + tile: P_X(j) V_j computed
  BAR_MMA_DONE = BAR_O_DONE + kMaxQTiles,
  BAR_O_STAGED = BAR_MMA_DONE + 1,        // + tile: the tile's O rows are in shared memory
  BAR_S_READ = BAR_O_STAGED + kMaxQTiles, // one-tile CTA: S(j) loaded by the softmax (128)
  BAR_COUNT = BAR_S_READ + 1
};
static_assert(BAR_COUNT <= 24, "barrier slots");

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

// Which keys a query may attend to ("FlashAttention 优化原理与实现要点解析" §7 causal mask and
// the padding and sliding-window masks §8 names): key j is allowed for query i when
// j < len (the batch's key length), j <= i (causal), j >= i - left (left >= 0) and
// j <= i + right (right >= 0). The allowed keys of one query form the interval [lo(i), hi(i)),
// and lo, hi never decrease with i.
// WINDOWED = false: no window and no per-batch key length (only causal and the ragged tail), so
// those terms fold away at compile time.
// Query i sits at key position i + offset (offset = Nk - Nq: the queries are the last Nq
// positions of the sequence, as when decoding against a longer key/value sequence).
template <bool WINDOWED>
struct KeyMask {
  int len, causal, left, right, offset;
  __device__ __forceinline__ int lo(int i) const {
    if constexpr (WINDOWED) return left >= 0 ? max(0, i + offset - left) : 0;
    return 0;
  }
  __device__ __forceinline__ int hi(int i) const {
    int z = len;
    if (causal) z = min(z, i + offset + 1);
    if constexpr (WINDOWED) {
      if (right >= 0) z = min(z, i + offset + right + 1);
    }
    return z;
  }
  // K/V tiles [j0, j1) that hold an allowed key of some row of Q tile qt (rows < Nq only);
  // j1 <= j0 when there is none.
  __device__ __forceinline__ void tile_range(int qt, int Nq, int& j0, int& j1) const {
    const int r0 = qt * BLOCK_M;
    const int r_last = min(r0 + BLOCK_M, Nq) - 1;
    const int a = lo(r0), z = r0 < Nq ? hi(r_last) : 0;
    if (z <= a) {
      j0 = 0;
      j1 = 0;
    } else {
      j0 = a / BLOCK_N;
      j1 = (z + BLOCK_N - 1) / BLOCK_N;
    }
  }
};

// ---------------------------------------------------------------------------------------------
template <int QT, int D, bool FP16, bool WINDOWED>
__global__ void __launch_bounds__((Cfg<QT, D>::kThreads), (Cfg<QT, D>::kMinBlocks))
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_o, void* __restrict__ o_ptr,
                  float* __restrict__ lse_ptr, int H, int Nq, int Nk, int causal,
                  float scale_log2, int heads_per_group, int window_left, int window_right,
                  const int* __restrict__ seqlens_k, int num_splits,
                  float* __restrict__ o_part, float* __restrict__ lse_part) {
  using L = SmemLayout<QT, D>;
  using C = Cfg<QT, D>;
  constexpr int kQTiles = QT;
  constexpr uint32_t kTmemO = C::kTmemO;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  const uint32_t smem_base = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = smem_base + L::kQ;
  const uint32_t sK = smem_base + L::kK;
  const uint32_t sV = smem_base + L::kV;
  auto bar = [&](int i) { return smem_base + L::kBars + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // Work unit from a 1-D grid. Heads are taken in groups of `heads_per_group` (sized on the
  // host so that a group's K and V stay resident in L2); within a group, units go Q block by
  // Q block across the group's heads, longest (causal) block first, so the CTAs in flight share
  // few heads and the long blocks start early.
  // With num_splits > 1 every Q block's K/V range is cut into num_splits consecutive parts,
  // one per CTA; the parts of a block are dispatched together.
  const int num_qblk = (Nq + kQTiles * BLOCK_M - 1) / (kQTiles * BLOCK_M);
  const int num_bh = gridDim.x / (num_qblk * num_splits);
  const int group_units = heads_per_group * num_qblk * num_splits;
  const int g = static_cast<int>(blockIdx.x) / group_units;
  const int rem = static_cast<int>(blockIdx.x) % group_units;
  const int g_size = min(heads_per_group, num_bh - g * heads_per_group);
  const int bh = g * heads_per_group + rem % g_size;
  const int r = rem / g_size / num_splits;
  const int split = (rem / g_size) % num_splits;
  const int qblk = causal ? num_qblk - 1 - r : r;
  const int b = bh / H, h = bh % H;
  KeyMask<WINDOWED> mask;
  mask.len = (WINDOWED && seqlens_k) ? min(max(seqlens_k[b], 0), Nk) : Nk;
  mask.causal = causal;
  mask.left = window_left;
  mask.right = window_right;
  mask.offset = Nk - Nq;
  // K/V tile ranges of tile A and tile B ([x0, x1), empty when x1 <= x0; a0 <= b0 and
  // a1 <= b1 when both are non-empty) and their union [u0, u1), which the producer streams.
  int a0, a1, b0, b1;
  mask.tile_range(kQTiles * qblk, Nq, a0, a1);
  if constexpr (QT == 2) {
    mask.tile_range(kQTiles * qblk + 1, Nq, b0, b1);
  } else {
    b0 = b1 = 0;   // no tile B
  }
  if (num_splits > 1) {
    // this CTA's part of the block's K/V tiles: [c0, c1)
    const int w0 = a1 > a0 ? a0 : b0, w1 = b1 > b0 ? b1 : a1;
    const int span = max(w1 - w0, 0);
    const int c0 = w0 + span * split / num_splits, c1 = w0 + span * (split + 1) / num_splits;
    a0 = max(a0, c0);
    a1 = min(a1, c1);
    b0 = max(b0, c0);
    b1 = min(b1, c1);
  }
  const bool a_any = a1 > a0, b_any = b1 > b0;
  const int u0 = a_any ? a0 : b0;
  const int u1 = b_any ? b1 : a1;
  const bool any_work = a_any || b_any;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(bar(BAR_Q_FULL), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(BAR_K_FULL + s), 1);
      ptx::mbar_init(bar(BAR_K_EMPTY + s), 1);
      ptx::mbar_init(bar(BAR_V_FULL + s), 1);
      ptx::mbar_init(bar(BAR_V_EMPTY + s), 1);
    }
    for (int x = 0; x < kQTiles; ++x) {
      ptx::mbar_init(bar(BAR_S_FULL + x), 1);
      ptx::mbar_init(bar(BAR_P_FULL + x), 128);
      ptx::mbar_init(bar(BAR_O_DONE + x), 1);
      ptx::mbar_init(bar(BAR_O_STAGED + x), 128);
    }
    ptx::mbar_init(bar(BAR_S_READ), 128);
    ptx::mbar_init(bar(BAR_MMA_DONE), 1);
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&tmem_base_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = tmem_base_slot;
  volatile int* abort_p = &abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    // K/V tiles u0, u0+1, ..., u1-1 go through the rings in order; load n of the sequence uses
    // stage n % kStages.
    if (lane == 0 && any_work) {
      ptx::prefetch_tensormap(&tm_q);
      ptx::prefetch_tensormap(&tm_k);
      ptx::prefetch_tensormap(&tm_v);
      ptx::prefetch_tensormap(&tm_o);
      ptx::mbar_arrive_expect_tx(bar(BAR_Q_FULL), kQTiles * L::kTile);
      for (int x = 0; x < kQTiles; ++x)
        for (int c = 0; c < D / BOX_COLS; ++c)
          ptx::tma_load_4d(sQ + x * L::kTile + c * kBoxBytes, &tm_q, bar(BAR_Q_FULL),
                           c * BOX_COLS, h, (kQTiles * qblk + x) * BLOCK_M, b);
      int k_issued = 0, v_issued = 0;
      for (int n = 0; n < u1 - u0; ++n) {
        const int s = n % kStages;
        const uint32_t ph = (n / kStages) & 1;
        const int kv_row0 = (u0 + n) * BLOCK_N;
        if (!ptx::wait_bounded(bar(BAR_K_EMPTY + s), ph ^ 1, abort_p, kWaitLimitNs)) {
          record_timeout(abort_p);
          break;
        }
        ptx::mbar_arrive_expect_tx(bar(BAR_K_FULL + s), L::kTile);
        for (int c = 0; c < D / BOX_COLS; ++c)
          ptx::tma_load_4d(sK + s * L::kTile + c * kBoxBytes, &tm_k, bar(BAR_K_FULL + s),
                           c * BOX_COLS, h, kv_row0, b);
        k_issued = n + 1;
        if (!ptx::wait_bounded(bar(BAR_V_EMPTY + s), ph ^ 1, abort_p, kWaitLimitNs)) {
          record_timeout(abort_p);
          break;
        }
        ptx::mbar_arrive_expect_tx(bar(BAR_V_FULL + s), L::kTile);
        for (int c = 0; c < D / BOX_COLS; ++c)
          ptx::tma_load_4d(sV + s * L::kTile + c * kBoxBytes, &tm_v, bar(BAR_V_FULL + s),
                           c * BOX_COLS, h, kv_row0, b);
        v_issued = n + 1;
      }
      // Leave no copy in flight: wait (bounded) for Q and for the last load into every stage.
      // On the normal path these phases completed long ago.
      ptx::wait_bounded(bar(BAR_Q_FULL), 0, abort_p, kWaitLimitNs);
      for (int n = (k_issued > kStages ? k_issued - kStages : 0); n < k_issued; ++n)
        ptx::wait_bounded(bar(BAR_K_FULL + n % kStages), (n / kStages) & 1, abort_p,
                          kWaitLimitNs);
      for (int n = (v_issued > kStages ? v_issued - kStages : 0); n < v_issued; ++n)
        ptx::wait_bounded(bar(BAR_V_FULL + n % kStages), (n / kStages) & 1, abort_p,
                          kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = ptx::idesc_f16(FP16, BLOCK_M, BLOCK_N, false);
      constexpr uint32_t idesc_pv = ptx::idesc_f16(FP16, BLOCK_M, D, true);
      auto wait = [&](int slot, uint32_t parity) {
        return ptx::wait_bounded(bar(slot), parity, abort_p, kWaitLimitNs);
      };
      // S_x(j) = Q_x K_j^T into the S columns of tile x (K_j sits in stage (j - u0) % kStages).
      auto issue_s = [&](int x, int j) {
        ptx::tc_fence_after_sync();
        const ptx::SmemDesc q_desc = ptx::smem_desc_sw128_split(sQ + x * L::kTile, 16, 1024);
        const ptx::SmemDesc k_desc =
            ptx::smem_desc_sw128_split(sK + ((j - u0) % kStages) * L::kTile, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // 16 elements (32 bytes) of d per MMA: 4 steps inside one 128-byte swizzle span,
          // then the next 64-column box.
          const uint32_t off = (kk / 4) * kBoxBytes + (kk % 4) * 32;
          ptx::mma_f16_ss(tmem + x * BLOCK_N, q_desc.at(off), k_desc.at(off), idesc_qk, kk > 0);
        }
        ptx::mma_commit(bar(BAR_S_FULL + x));
      };
      // O_x += P_x(j) V_j: A = P_x from TMEM (16 keys = 8 columns per MMA), B = V tile,
      // MN-major (d contiguous): 16 keys = 16 rows of 128 bytes per MMA, LBO = next 64-column box.
      // The first P V of a tile overwrites O instead of accumulating.
      auto issue_pv = [&](int x, int j, bool first) {
        ptx::tc_fence_after_sync();
        const ptx::SmemDesc v_desc =
            ptx::smem_desc_sw128_split(sV + ((j - u0) % kStages) * L::kTile, kBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < BLOCK_N / 16; ++kk)
          ptx::mma_f16_ts(tmem + kTmemO + x * D,
                          tmem + (C::kSeparateP ? C::kTmemP : x * BLOCK_N) + kk * 8,
                          v_desc.at(kk * 16 * 128), idesc_pv, (!first || kk > 0) ? 1u : 0u);
        ptx::mma_commit(bar(BAR_O_DONE + x));
      };

      auto on_a = [&](int j) { return a0 <= j && j < a1; };
      auto on_b = [&](int j) { return QT == 2 && b0 <= j && j < b1; };
      // K_j / V_j are load number j - u0 of the sequence.
      auto wait_k = [&](int j) {
        return wait(BAR_K_FULL + (j - u0) % kStages, ((j - u0) / kStages) & 1);
      };
      auto wait_v = [&](int j) {
        return wait(BAR_V_FULL + (j - u0) % kStages, ((j - u0) / kStages) & 1);
      };
      bool ok = true;
      if (any_work) {
        ok = wait(BAR_Q_FULL, 0) && wait_k(u0);
        if (ok) {
          if (on_a(u0)) issue_s(0, u0);
          if (on_b(u0)) issue_s(1, u0);
          ptx::mma_commit(bar(BAR_K_EMPTY + 0));
        }
      }
      if constexpr (C::kSeparateP) {
        // One tile, P in columns of its own: S(j+1) is issued once the softmax has loaded S(j)
        // (S_READ), so it is computed while that softmax runs; P(j) V_j once P(j) is stored.
        // The softmax waits for P(j-1) V_{j-1} (O_DONE) before it writes P(j) or rescales O.
        for (int j = u0; ok && any_work && j < u1; ++j) {
          const int s = (j - u0) % kStages;
          if (j + 1 < u1) {
            if (!wait_k(j + 1) || !wait(BAR_S_READ, (j - a0) & 1)) { ok = false; break; }
            issue_s(0, j + 1);
            ptx::mma_commit(bar(BAR_K_EMPTY + (j + 1 - u0) % kStages));
          }
          if (!wait_v(j) || !wait(BAR_P_FULL + 0, (j - a0) & 1)) { ok = false; break; }
          issue_pv(0, j, j == a0);
          ptx::mma_commit(bar(BAR_V_EMPTY + s));
        }
      }
      // Per K/V tile j: P_A(j) V_j, S_A(j+1), P_B(j) V_j, S_B(j+1). The softmax of one tile
      // runs while the tensor pipe works on the other.
      for (int j = u0; !C::kSeparateP && ok && any_work && j < u1; ++j) {
        const int s = (j - u0) % kStages;
        const bool next = j + 1 < u1;
        if (!wait_v(j)) { ok = false; break; }
        if (on_a(j)) {
          if (!wait(BAR_P_FULL + 0, (j - a0) & 1)) { ok = false; break; }
          issue_pv(0, j, j == a0);
        }
        if (next && !wait_k(j + 1)) { ok = false; break; }
        if (on_a(j + 1)) issue_s(0, j + 1);
        if (on_b(j)) {
          if (!wait(BAR_P_FULL + 1, (j - b0) & 1)) { ok = false; break; }
          issue_pv(1, j, j == b0);
        }
        ptx::mma_commit(bar(BAR_V_EMPTY + s));
        if (on_b(j + 1)) issue_s(1, j + 1);
        if (next) ptx::mma_commit(bar(BAR_K_EMPTY + (j + 1 - u0) % kStages));
      }
      if (!ok) record_timeout(abort_p);
      // Every MMA this thread issued has completed before TMEM can be released.
      ptx::mma_commit(bar(BAR_MMA_DONE));
      wait(BAR_MMA_DONE, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    const int x = (warp - 2) / 4;                       // Q tile: 0 = A, 1 = B
    const int quarter = warp & 3;                       // TMEM lanes [32q, 32q+32)
    const int row = quarter * 32 + lane;                // query row within the tile
    const int qt = kQTiles * qblk + x;                  // global Q tile index
    const int q_idx = qt * BLOCK_M + row;               // query index (position - offset)
    const int x0 = x ? b0 : a0, x1 = x ? b1 : a1;       // this tile's K/V tiles [x0, x1)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + x * BLOCK_N;
    // where P_x(j) goes: columns of its own (one-tile CTA) or over S_x
    const uint32_t tP = C::kSeparateP ? tmem + lane_off + C::kTmemP : tS;
    const uint32_t tO = tmem + lane_off + kTmemO + x * D;
    const bool scale_pos = scale_log2 > 0.f;
    // This row's allowed keys [row_lo, row_hi); a K/V tile starting at k0 needs no per-element
    // mask when full_lo <= k0 and k0 + BLOCK_N <= full_hi (inside every row's interval).
    const int row_lo = mask.lo(q_idx), row_hi = mask.hi(q_idx);
    const int full_lo = mask.lo(qt * BLOCK_M + BLOCK_M - 1), full_hi = mask.hi(qt * BLOCK_M);
    float m = -INFINITY;   // exponent offset in use, log2 units of scaled scores
    float l = 0.f;         // sum of 2^(scaled score - m) over the keys seen so far
    bool ok = true;

    for (int j = x0; j < x1; ++j) {
      if (!ptx::wait_bounded_warp(bar(BAR_S_FULL + x), (j - x0) & 1, abort_p, kWaitLimitNs)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after_sync();
      uint32_t sr[BLOCK_N / 32][32];
#pragma unroll
      for (int c = 0; c < BLOCK_N / 32; ++c) ptx::tmem_ld_32x32b_x32(tS + c * 32, sr[c]);
      ptx::tmem_wait_ld();
      if constexpr (C::kSeparateP) {
        // S_x(j) is in registers: the MMA thread may compute S_x(j+1) over it
        ptx::tc_fence_before_sync();
        ptx::mbar_arrive(bar(BAR_S_READ));
      }
      float s[BLOCK_N];
#pragma unroll
      for (int c = 0; c < BLOCK_N / 32; ++c) {
        ptx::reg_fence(sr[c]);
#pragma unroll
        for (int t = 0; t < 32; ++t) s[c * 32 + t] = __uint_as_float(sr[c][t]);
      }

      const int k0 = j * BLOCK_N;
      if (!scale_pos) {
        // Non-positive scale: scale first, so that the maximum below is the maximum of the
        // scaled scores.
#pragma unroll
        for (int t = 0; t < BLOCK_N; t += 2)
          ptx::mul2(s[t], s[t + 1], s[t], s[t + 1], scale_log2, scale_log2);
      }
      if (k0 < full_lo || k0 + BLOCK_N > full_hi) {
        const int lo = row_lo - k0, hi = row_hi - k0;   // keys k0 + [lo, hi) are allowed
        if constexpr (WINDOWED) {
#pragma unroll
          for (int t = 0; t < BLOCK_N; ++t)
            if (t < lo || t >= hi) s[t] = -INFINITY;
        } else {
#pragma unroll
          for (int t = 0; t < BLOCK_N; ++t)
            if (t >= hi) s[t] = -INFINITY;
        }
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int t = 0; t < BLOCK_N; t += 8) {
        mx[0] = ptx::max3(mx[0], s[t + 0], s[t + 1]);
        mx[1] = ptx::max3(mx[1], s[t + 2], s[t + 3]);
        mx[2] = ptx::max3(mx[2], s[t + 4], s[t + 5]);
        mx[3] = ptx::max3(mx[3], s[t + 6], s[t + 7]);
      }
      const float mt = fmaxf(ptx::max3(mx[0], mx[1], mx[2]), mx[3]);
      const float m_tile = scale_pos ? mt * scale_log2 : mt;
      float alpha = 1.f;
      const bool rescale = __any_sync(0xffffffffu, m_tile > m + kRescaleLog2);
      if (rescale) {
        // Move every row of this warp to its running maximum; l now, O below.
        const float m_new = fmaxf(m, m_tile);
        alpha = ptx::exp2_approx(m - (m_new == -INFINITY ? 0.f : m_new));
        l *= alpha;
        m = m_new;
      }
      const float m_use = (m == -INFINITY) ? 0.f : m;
      if constexpr (C::kSeparateP) {
        // P_x(j-1) V_{j-1} reads the P columns and accumulates into O: both must be done
        // before P_x(j) is written or O rescaled (S_x(j) no longer implies it here).
        if (j > x0) {
          if (!ptx::wait_bounded_warp(bar(BAR_O_DONE + x), (j - 1 - x0) & 1, abort_p,
                                      kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after_sync();
        }
      }

      // P_x(j) = 2^(scaled score - m) -> TMEM (over the first 64 columns of S_x, or the P
      // columns of the one-tile CTA), 32 keys (16 columns) at a time: column c holds keys 2c
      // (low half) and 2c + 1 (high half), rounded to the input type.
      // exponent argument: s * scale_log2 - m_use (positive scale, folded into one FMA) or
      // s - m_use (s already scaled)
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int c = 0; c < BLOCK_N / 32; ++c) {
        uint32_t pr[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          float e0, e1;
          if (scale_pos)
            ptx::fma2(e0, e1, s[32 * c + 2 * t], s[32 * c + 2 * t + 1], scale_log2, scale_log2,
                      -m_use, -m_use);
          else
            ptx::add2(e0, e1, s[32 * c + 2 * t], s[32 * c + 2 * t + 1], -m_use, -m_use);
          const float p0 = ptx::exp2_approx(e0);
          const float p1 = ptx::exp2_approx(e1);
          ptx::add2(rs0, rs1, rs0, rs1, p0, p1);
          pr[t] = pack2<FP16>(p0, p1);
        }
        ptx::tmem_st_32x32b_x16(tP + c * 16, pr);
      }
      l += rs0 + rs1;

      if (rescale && j > x0) {
        // P_x(j-1) V_{j-1} has completed: it was issued before S_x(j) (one-tile CTA: waited
        // for above). The whole O row is loaded at once (the registers of S are free by
        // now), so the rescale costs one TMEM round trip instead of one per 32 columns.
        uint32_t orr[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) ptx::tmem_ld_32x32b_x32(tO + c * 32, orr[c]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          ptx::reg_fence(orr[c]);
#pragma unroll
          for (int t = 0; t < 32; t += 2) {
            float a0 = __uint_as_float(orr[c][t]), a1 = __uint_as_float(orr[c][t + 1]);
            ptx::mul2(a0, a1, a0, a1, alpha, alpha);
            orr[c][t] = __float_as_uint(a0);
            orr[c][t + 1] = __float_as_uint(a1);
          }
          ptx::tmem_st_32x32b_x32(tO + c * 32, orr[c]);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before_sync();
      ptx::mbar_arrive(bar(BAR_P_FULL + x));
    }

    // ---------------------------------------------------------------- epilogue
    // One split: O (input type) and LSE go straight to the outputs. Several splits: this
    // CTA's part, normalised by its own l, goes to the fp32 workspace with its own LSE;
    // fa_merge_kernel combines the parts.
    const bool valid = q_idx < Nq;
    const int64_t row_id = static_cast<int64_t>(bh) * Nq + q_idx;   // (b, h, q)
    const int64_t part_row = static_cast<int64_t>(split) * num_bh * Nq + row_id;
    uint16_t* out_row = static_cast<uint16_t*>(o_ptr) +
                        ((static_cast<int64_t>(b) * Nq + q_idx) * H + h) * D;
    if (x1 <= x0) {
      // No allowed key for this tile (in this part): O = 0 and LSE = -inf, no TMEM access.
      if (valid) {
        if (num_splits == 1) {
          uint4* dst = reinterpret_cast<uint4*>(out_row);
#pragma unroll
          for (int t = 0; t < D / 8; ++t) dst[t] = make_uint4(0, 0, 0, 0);
          lse_ptr[row_id] = -INFINITY;
        } else {
          float4* dst = reinterpret_cast<float4*>(o_part + part_row * D);
#pragma unroll
          for (int t = 0; t < D / 4; ++t) dst[t] = make_float4(0.f, 0.f, 0.f, 0.f);
          lse_part[part_row] = -INFINITY;
        }
      }
    } else if (ok && ptx::wait_bounded_warp(bar(BAR_O_DONE + x), (x1 - x0 - 1) & 1, abort_p,
                                       kWaitLimitNs)) {
      ptx::tc_fence_after_sync();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      // One split: the normalised O row goes into tile x's Q buffer (no MMA reads it any more:
      // its last S finished before the last P V), laid out as the TMA boxes of the O tensor
      // map (128-byte swizzle: 16-byte chunk k of row r at chunk k ^ (r % 8)); one thread then
      // stores the whole 128-row tile with TMA, which leaves out rows at or past Nq.
      const uint32_t staging = sQ + x * L::kTile;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orr[32];
        ptx::tmem_ld_32x32b_x32(tO + c * 32, orr);
        ptx::tmem_wait_ld();
        ptx::reg_fence(orr);
        if (num_splits == 1) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int col0 = c * 32 + t * 8;
            const uint32_t addr = staging + (col0 / BOX_COLS) * kBoxBytes + row * 128 +
                                  ((((col0 % BOX_COLS) / 8) ^ (row & 7)) << 4);
            ptx::st_shared_v4(addr,
                              pack2<FP16>(__uint_as_float(orr[8 * t + 0]) * inv_l,
                                          __uint_as_float(orr[8 * t + 1]) * inv_l),
                              pack2<FP16>(__uint_as_float(orr[8 * t + 2]) * inv_l,
                                          __uint_as_float(orr[8 * t + 3]) * inv_l),
                              pack2<FP16>(__uint_as_float(orr[8 * t + 4]) * inv_l,
                                          __uint_as_float(orr[8 * t + 5]) * inv_l),
                              pack2<FP16>(__uint_as_float(orr[8 * t + 6]) * inv_l,
                                          __uint_as_float(orr[8 * t + 7]) * inv_l));
          }
        } else if (valid) {
          float4* dst = reinterpret_cast<float4*>(o_part + part_row * D + c * 32);
#pragma unroll
          for (int t = 0; t < 8; ++t)
            dst[t] = make_float4(__uint_as_float(orr[4 * t + 0]) * inv_l,
                                 __uint_as_float(orr[4 * t + 1]) * inv_l,
                                 __uint_as_float(orr[4 * t + 2]) * inv_l,
                                 __uint_as_float(orr[4 * t + 3]) * inv_l);
        }
      }
      if (num_splits == 1) {
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(bar(BAR_O_STAGED + x));
        if (row == 0) {
          if (ptx::wait_bounded(bar(BAR_O_STAGED + x), 0, abort_p, kWaitLimitNs)) {
#pragma unroll
            for (int bx = 0; bx < D / BOX_COLS; ++bx)
              ptx::tma_store_4d(&tm_o, staging + bx * kBoxBytes, bx * BOX_COLS, h, qt * BLOCK_M,
                                b);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_read0();   // shared memory stays valid until it has been read
          } else {
            record_timeout(abort_p);
          }
        }
      }
      if (valid) {
        const float lse_row = (m + __log2f(l)) * 0.69314718055994530942f;
        if (num_splits == 1)
          lse_ptr[row_id] = lse_row;
        else
          lse_part[part_row] = lse_row;
      }
    } else {
      record_timeout(abort_p);
    }
  }

  // ------------------------------------------------------------------ teardown
  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------------
// Merge of split K/V parts ("FlashAttention 优化原理与实现要点解析" §4.2: per-block statistics
// merged into the global ones). Part s of a row holds O_s (normalised by its own l_s) and
// LSE_s = m_s + ln l_s. Then LSE = ln sum_s e^{LSE_s} and O = sum_s e^{LSE_s - LSE} O_s.
// One warp per (b, h, q) row; lane t owns D / 32 consecutive columns.
template <int D, bool FP16>
__global__ void __launch_bounds__(256)
    fa_merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                    void* __restrict__ o_ptr, float* __restrict__ lse_ptr, int H, int Nq,
                    long long rows, int num_splits) {
  constexpr int E = D / 32;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32;
  if (row >= rows) return;
  const int lane = threadIdx.x % 32;
  float mx = -INFINITY;
  for (int s = lane; s < num_splits; s += 32) mx = fmaxf(mx, lse_part[s * rows + row]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float sum = 0.f;
  if (mx != -INFINITY)
    for (int s = lane; s < num_splits; s += 32) sum += expf(lse_part[s * rows + row] - mx);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float lse_row = mx == -INFINITY ? -INFINITY : mx + logf(sum);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < num_splits; ++s) {
      const float ls = lse_part[s * rows + row];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - lse_row);
      const float* src = o_part + (s * rows + row) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(w, src[e], acc[e]);
    }
  }
  const long long bh = row / Nq;
  const int q = static_cast<int>(row % Nq);
  const long long b = bh / H, h = bh % H;
  uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(o_ptr) +
                                              ((b * Nq + q) * H + h) * D + lane * E);
#pragma unroll
  for (int e = 0; e < E; e += 2) dst[e / 2] = pack2<FP16>(acc[e], acc[e + 1]);
  if (lane == 0) lse_ptr[row] = lse_row;
}

template <int QT, int D, bool FP16, bool WINDOWED>
cudaError_t launch_impl(const FwdParams& p, cudaStream_t stream) {
  auto kernel = fa_fwd_kernel<QT, D, FP16, WINDOWED>;
  const size_t smem = SmemLayout<QT, D>::kDynamic;
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const long long num_qblk = (p.Nq + QT * BLOCK_M - 1) / (QT * BLOCK_M);
  const long long bh = static_cast<long long>(p.B) * p.H;
  const dim3 grid(static_cast<unsigned>(num_qblk * bh * p.num_splits));
  // Heads per dispatch group: K and V of a group within 32 MiB, a quarter of L2, so that they
  // stay resident beside the streamed Q tiles and O rows while every Q block of the group
  // reads them (measured: 64 MiB groups read K and V 1.4-2.3 times from DRAM, 32 MiB groups
  // once, at the same speed; 16 MiB groups were slower on long causal sequences).
  const long long kv_bytes_per_head = 4ll * p.Nk * p.d;
  const int heads_per_group =
      static_cast<int>(std::max(1ll, std::min(bh, (32ll << 20) / kv_bytes_per_head)));
  kernel<<<grid, Cfg<QT, D>::kThreads, smem, stream>>>(p.tm_q, p.tm_k, p.tm_v, p.tm_o, p.o, p.lse, p.H, p.Nq, p.Nk,
                                           p.causal, p.scale_log2, heads_per_group,
                                           p.window_left, p.window_right, p.seqlens_k,
                                           p.num_splits, p.o_part, p.lse_part);
  err = cudaGetLastError();
  if (err != cudaSuccess || p.num_splits == 1) return err;
  const long long rows = bh * p.Nq;
  fa_merge_kernel<D, FP16><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
      p.o_part, p.lse_part, p.o, p.lse, p.H, p.Nq, rows, p.num_splits);
  return cudaGetLastError();
}

}  // namespace

template <bool WINDOWED>
cudaError_t launch_dtype(const FwdParams& p, cudaStream_t stream) {
  if (p.d == 64) {
    // d = 64 (not split): one Q tile per CTA, P in columns of its own, two CTAs per SM. Against
    // the two-tile CTA: B=4 H=16 N=1K 39 -> 34 us; B=2 H=16 N=8K causal 359 -> 291 us,
    // non-causal 671 -> 557 us.
    if (p.num_splits == 1)
      return p.fp16 ? launch_impl<1, 64, true, WINDOWED>(p, stream)
                    : launch_impl<1, 64, false, WINDOWED>(p, stream);
    return p.fp16 ? launch_impl<2, 64, true, WINDOWED>(p, stream)
                  : launch_impl<2, 64, false, WINDOWED>(p, stream);
  }
  return p.fp16 ? launch_impl<2, 128, true, WINDOWED>(p, stream)
                : launch_impl<2, 128, false, WINDOWED>(p, stream);
}

cudaError_t launch_fwd(const FwdParams& p, cudaStream_t stream) {
  const bool windowed = p.window_left >= 0 || p.window_right >= 0 || p.seqlens_k != nullptr;
  return windowed ? launch_dtype<true>(p, stream) : launch_dtype<false>(p, stream);
}

namespace {

// Diagnostic: one thread waits, with the kernels' own bounded wait, on an mbarrier that nothing
// ever arrives on, and records the timeout in the error word exactly as the attention kernels
// do. It exercises the failure path (wait runs out -> error word -> host) without a fault.
__global__ void __launch_bounds__(32) fa_selftest_wait_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t never;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(ptx::smem_addr(&never), 1);
    ptx::fence_barrier_init();
    if (!ptx::wait_bounded(ptx::smem_addr(&never), 0, &abort_flag, limit_ns))
      record_timeout(&abort_flag);
  }
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream) {
  fa_selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
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
