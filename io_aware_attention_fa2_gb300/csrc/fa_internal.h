// fa_internal.h -- declarations shared by the translation units of the CUDA library
// (fa_api.cpp: argument checks, tensor maps, C ABI; fa_fwd_kernel.cu, fa_bwd_kernel.cu:
// kernels and launch; fa_noalloc.cu: the entry point with a built-in workspace).
// Not part of the public ABI (that is include/fa.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// Tile shape of one work unit: BLOCK_M query rows against BLOCK_N keys per K/V tile.
constexpr int BLOCK_M = 128;
constexpr int BLOCK_N = 128;
// A TMA box is BOX_ROWS tokens x BOX_COLS 16-bit elements (one 128-byte swizzle span per row).
constexpr int BOX_ROWS = 128;
constexpr int BOX_COLS = 64;
// Most K/V parts a split forward may use.
constexpr int MAX_SPLITS = 128;

struct FwdParams {
  CUtensorMap tm_q;   // [B, N, H, d] viewed as 4-D (d, H, N, B); box (64, 1, 128, 1)
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_o;   // o as a 4-D map like tm_q (the epilogue stores O tiles through it)
  void* o;            // [B, N, H, d], same storage type as q
  float* lse;         // [B, H, N]
  int B, H, d;
  int Nq, Nk;         // queries (q, o, lse) and keys (k, v); Nk >= Nq, queries are the last Nq
  int num_splits;     // >= 1: parts each (b, h, Q block)'s K/V range is cut into
  float* o_part;      // num_splits > 1: fp32 [num_splits, B, H, Nq, d] partial O (workspace)
  float* lse_part;    // num_splits > 1: fp32 [num_splits, B, H, Nq] partial LSE (workspace)
  int causal;
  int window_left;    // key j visible to query i only if j >= i - window_left (< 0: no bound)
  int window_right;   // ... and j <= i + window_right (< 0: no bound)
  const int* seqlens_k;  // device int32 [B]: keys at or past seqlens_k[b] are masked; or null
  int fp16;           // 0: bf16, 1: fp16
  float scale_log2;   // scale * log2(e)
};

// Enqueue the forward kernel. Returns a CUDA error (cudaSuccess when enqueued).
cudaError_t launch_fwd(const FwdParams& p, cudaStream_t stream);

// Device error word of the current device: read (after synchronising `stream`) and clear.
cudaError_t read_and_clear_device_error(cudaStream_t stream, int* value);

// The bounded-wait self-test kernel (a wait on an mbarrier nothing arrives on).
cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream);

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;   // [B, N, H, d] as in FwdParams
  const void* o;        // [B, N, H, d] forward output
  const void* dout;     // [B, N, H, d] upstream gradient
  const float* lse;     // [B, H, N] from the forward
  void* dq;             // [B, N, H, d]
  void* dk;
  void* dv;
  float* dq_acc;        // workspace: fp32 [B, H, N, d], sum over key blocks of dS K
  float* dpre;          // workspace: fp32 [B, H, N], D = rowsum(dO * O)
  int B, H, N, d;
  int causal;
  int window_left;      // as in FwdParams (queries and keys share positions here)
  int window_right;
  const int* seqlens_k; // device int32 [B] or null, as in FwdParams
  int fp16;
  float scale;
};

// Every host-side check fa_fwd_splitkv makes except those of its workspace argument: the
// FA_* code it would return for these arguments (nothing is enqueued).
int check_splitkv_args(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int Nq, int Nk, int d, const int* seqlens_k, float scale,
                       int dtype, int num_splits);

// Enqueue the backward (pre-kernel, main kernel, post-kernel).
cudaError_t launch_bwd(const BwdParams& p, cudaStream_t stream);
// The backward kernels' error word of the current device: read and clear (no synchronisation).
cudaError_t read_and_clear_bwd_error(int* value);

}  // namespace fa
