// fa_api.cpp -- the C ABI of include/fa.h: argument checks, TMA tensor maps, launch.
//
// Host-detected errors return before anything is enqueued. No C++ exception crosses the ABI.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_arch_ok[kMaxDevices];   // 0 unknown, 1 sm_103, -1 other

int check_arch(int* device) {
  if (cudaGetDevice(device) != cudaSuccess) return FA_ERR_CUDA;
  if (*device < 0 || *device >= kMaxDevices) return FA_ERR_CUDA;
  int state = g_arch_ok[*device].load(std::memory_order_relaxed);
  if (state == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *device) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *device) !=
            cudaSuccess)
      return FA_ERR_CUDA;
    state = (major == 10 && minor == 3) ? 1 : -1;
    g_arch_ok[*device].store(state, std::memory_order_relaxed);
  }
  return state == 1 ? FA_OK : FA_ERR_ARCH;
}

bool overlaps(const void* a, uint64_t a_bytes, const void* b, uint64_t b_bytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

// [B, N, H, d] 16-bit tensor as a 4-D TMA map (d, H, N, B) with box (64, 1, 128, 1) and the
// 128-byte swizzle. Rows past N read as zeros.
bool encode_bnhd(CUtensorMap* map, const void* base, int B, int H, int N, int d, bool fp16) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2,
                                 (cuuint64_t)N * H * d * 2};
  const cuuint32_t box[4] = {(cuuint32_t)fa::BOX_COLS, 1, (cuuint32_t)fa::BOX_ROWS, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

int fa_abi_version(void) { return 1; }

const char* fa_error_string(int code) {
  switch (code) {
    case FA_OK: return "success";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_SHAPE: return "unsupported shape (B, H, N >= 1; d in {64, 128}; size overflow)";
    case FA_ERR_DTYPE: return "dtype is not FA_BF16 or FA_FP16";
    case FA_ERR_ALIGN:
      return "misaligned pointer (q, k, v, o: 16 bytes; lse, seqlens_k: 4 bytes)";
    case FA_ERR_ALIAS: return "an output overlaps an input, seqlens_k or the other output";
    case FA_ERR_ARCH: return "the current device is not sm_103 (GB300)";
    case FA_ERR_LAUNCH: return "kernel launch failed";
    case FA_ERR_TIMEOUT: return "a kernel wait ran past its limit";
    case FA_ERR_SCALE: return "scale is not finite";
    case FA_ERR_CUDA: return "a CUDA runtime or driver call failed";
    default: return "unknown status";
  }
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
           int N, int d, int causal, float scale, int dtype, fa_stream_t stream) {
  return fa_fwd_masked(q, k, v, o, lse, B, H, N, d, causal, -1, -1, nullptr, scale, dtype,
                       stream);
}

int fa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                  int H, int N, int d, int causal, int window_left, int window_right,
                  const int* seqlens_k, float scale, int dtype, fa_stream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return FA_ERR_SHAPE;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!isfinite(scale)) return FA_ERR_SCALE;
  // Sizes: elements must fit int64; the grid is one CTA per (b, h, 256-row Q block), at most
  // 2^31 - 1 CTAs.
  const uint64_t bh = (uint64_t)B * (uint64_t)H;
  if (bh >= (1ull << 31) || bh * (uint64_t)((N + 255) / 256) >= (1ull << 31))
    return FA_ERR_SHAPE;
  const uint64_t elems = bh * (uint64_t)N * (uint64_t)d;
  if (elems > (1ull << 62) / 2) return FA_ERR_SHAPE;
  const uint64_t t_bytes = elems * 2, lse_bytes = bh * (uint64_t)N * 4;
  for (const void* p : {q, k, v, static_cast<const void*>(o)})
    if (reinterpret_cast<uintptr_t>(p) % 16) return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) % 4) return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(seqlens_k) % 4) return FA_ERR_ALIGN;
  if (seqlens_k && (overlaps(seqlens_k, (uint64_t)B * 4, o, t_bytes) ||
                    overlaps(seqlens_k, (uint64_t)B * 4, lse, lse_bytes)))
    return FA_ERR_ALIAS;
  for (const void* in : {q, k, v})
    if (overlaps(o, t_bytes, in, t_bytes) || overlaps(lse, lse_bytes, in, t_bytes))
      return FA_ERR_ALIAS;
  if (overlaps(o, t_bytes, lse, lse_bytes)) return FA_ERR_ALIAS;

  int device = 0;
  int rc = check_arch(&device);
  if (rc != FA_OK) return rc;

  fa::FwdParams p;
  const bool fp16 = dtype == FA_FP16;
  if (!encode_bnhd(&p.tm_q, q, B, H, N, d, fp16) || !encode_bnhd(&p.tm_k, k, B, H, N, d, fp16) ||
      !encode_bnhd(&p.tm_v, v, B, H, N, d, fp16))
    return FA_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.N = N;
  p.d = d;
  p.causal = causal ? 1 : 0;
  p.window_left = window_left < 0 ? -1 : window_left;
  p.window_right = window_right < 0 ? -1 : window_right;
  p.seqlens_k = seqlens_k;
  p.fp16 = fp16 ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  if (fa::launch_fwd(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return FA_OK;
}

int fa_get_device_error(fa_stream_t stream) {
  int value = 0;
  if (fa::read_and_clear_device_error(reinterpret_cast<cudaStream_t>(stream), &value) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  return value == 0 ? FA_OK : FA_ERR_TIMEOUT;
}

}  // extern "C"
