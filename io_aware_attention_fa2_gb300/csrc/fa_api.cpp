// fa_api.cpp -- the C ABI of include/fa.h: argument checks, TMA tensor maps, launch.
//
// Host-detected errors return before anything is enqueued. No C++ exception crosses the ABI.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <initializer_list>
#include <mutex>
#include <vector>

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

// Every non-null pointer must be device (or managed) memory usable by `device`: a host or
// unknown address would make the kernels fault, so it is refused before anything is enqueued.
int check_device_ptrs(int device, std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs) {
    if (!p) continue;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
      cudaGetLastError();   // not sticky; leave no error behind for the caller
      return FA_ERR_POINTER;
    }
    if (a.type == cudaMemoryTypeManaged) continue;
    if (a.type != cudaMemoryTypeDevice || a.device != device) return FA_ERR_POINTER;
  }
  return FA_OK;
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
    case FA_ERR_SHAPE:
      return "unsupported shape (B, H, Nq >= 1; Nk >= Nq; d in {64, 128}; 1 <= num_splits <= "
             "128; size overflow)";
    case FA_ERR_DTYPE: return "dtype is not FA_BF16 or FA_FP16";
    case FA_ERR_ALIGN:
      return "misaligned pointer (q, k, v, o: 16 bytes; lse, seqlens_k: 4 bytes)";
    case FA_ERR_ALIAS: return "an output overlaps an input, seqlens_k or the other output";
    case FA_ERR_ARCH: return "the current device is not sm_103 (GB300)";
    case FA_ERR_LAUNCH: return "kernel launch failed";
    case FA_ERR_TIMEOUT: return "a kernel wait ran past its limit";
    case FA_ERR_SCALE: return "scale is not finite";
    case FA_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case FA_ERR_WORKSPACE: return "workspace smaller than fa_fwd_splitkv_workspace_size()";
    case FA_ERR_POINTER:
      return "a device-side argument is not device memory of the current device";
    default: return "unknown status";
  }
}

}  // extern "C"

namespace {

// Host-side checks shared by every forward entry point (nothing is enqueued).
// check_workspace = false skips the checks of the workspace argument (the caller supplies a
// workspace of its own afterwards).
int check_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                  int H, int Nq, int Nk, int d, int dtype, float scale, const int* seqlens_k,
                  int num_splits, void* workspace, size_t workspace_bytes,
                  bool inputs_written = false, bool check_workspace = true) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  if (B < 1 || H < 1 || Nq < 1 || Nk < Nq || (d != 64 && d != 128)) return FA_ERR_SHAPE;
  if (num_splits < 1 || num_splits > fa::MAX_SPLITS) return FA_ERR_SHAPE;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!isfinite(scale)) return FA_ERR_SCALE;
  // Sizes: elements must fit int64; the grid is one CTA per (b, h, 256-row Q block, K/V part),
  // at most 2^31 - 1 CTAs.
  const uint64_t bh = (uint64_t)B * (uint64_t)H;
  if (bh >= (1ull << 31) ||
      bh * (uint64_t)((Nq + 255) / 256) * (uint64_t)num_splits >= (1ull << 31))
    return FA_ERR_SHAPE;
  const uint64_t k_elems = bh * (uint64_t)Nk * (uint64_t)d;
  if (k_elems > (1ull << 62) / 2) return FA_ERR_SHAPE;
  const uint64_t q_bytes = bh * (uint64_t)Nq * d * 2, k_bytes = k_elems * 2;
  const uint64_t lse_bytes = bh * (uint64_t)Nq * 4;
  const uint64_t ws_need = fa_fwd_splitkv_workspace_size(B, H, Nq, d, num_splits);
  if (!check_workspace) workspace = nullptr;
  if (num_splits > 1 && check_workspace) {
    if (!workspace) return FA_ERR_NULL;
    if (workspace_bytes < ws_need) return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 16) return FA_ERR_ALIGN;
  }
  for (const void* p : {q, k, v, static_cast<const void*>(o)})
    if (reinterpret_cast<uintptr_t>(p) % 16) return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) % 4) return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(seqlens_k) % 4) return FA_ERR_ALIGN;
  struct Span { const void* p; uint64_t n; };
  const Span ins[] = {{q, q_bytes}, {k, k_bytes}, {v, k_bytes},
                      {seqlens_k, seqlens_k ? (uint64_t)B * 4 : 0}};
  const Span outs[] = {{o, q_bytes}, {lse, lse_bytes},
                       {num_splits > 1 ? workspace : nullptr, num_splits > 1 ? ws_need : 0}};
  for (const Span& out : outs) {
    if (!out.p) continue;
    for (const Span& in : ins)
      if (in.p && overlaps(out.p, out.n, in.p, in.n)) return FA_ERR_ALIAS;
  }
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (outs[i].p && outs[j].p && overlaps(outs[i].p, outs[i].n, outs[j].p, outs[j].n))
        return FA_ERR_ALIAS;
  // the host-buffer entry points copy into the input buffers, so these may not share memory
  if (inputs_written)
    for (int i = 0; i < 3; ++i)
      for (int j = i + 1; j < 3; ++j)
        if (overlaps(ins[i].p, ins[i].n, ins[j].p, ins[j].n)) return FA_ERR_ALIAS;
  int device = 0;
  const int rc = check_arch(&device);
  if (rc != FA_OK) return rc;
  return check_device_ptrs(device, {q, k, v, o, lse, seqlens_k,
                                    num_splits > 1 ? workspace : nullptr});
}

// Shared checks and launch of every forward entry point.
int run_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Nq, int Nk, int d, int causal, int window_left, int window_right,
                const int* seqlens_k, float scale, int dtype, int num_splits, void* workspace,
                size_t workspace_bytes, fa_stream_t stream) {
  const int rc = check_forward(q, k, v, o, lse, B, H, Nq, Nk, d, dtype, scale, seqlens_k,
                               num_splits, workspace, workspace_bytes);
  if (rc != FA_OK) return rc;
  const uint64_t bh = (uint64_t)B * (uint64_t)H;

  fa::FwdParams p;
  const bool fp16 = dtype == FA_FP16;
  if (!encode_bnhd(&p.tm_q, q, B, H, Nq, d, fp16) || !encode_bnhd(&p.tm_k, k, B, H, Nk, d, fp16) ||
      !encode_bnhd(&p.tm_v, v, B, H, Nk, d, fp16) || !encode_bnhd(&p.tm_o, o, B, H, Nq, d, fp16))
    return FA_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.d = d;
  p.causal = causal ? 1 : 0;
  p.window_left = window_left < 0 ? -1 : window_left;
  p.window_right = window_right < 0 ? -1 : window_right;
  p.seqlens_k = seqlens_k;
  p.fp16 = fp16 ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.num_splits = num_splits;
  p.o_part = num_splits > 1 ? static_cast<float*>(workspace) : nullptr;
  p.lse_part = num_splits > 1 ? static_cast<float*>(workspace) + bh * (uint64_t)Nq * d * num_splits
                              : nullptr;
  if (fa::launch_fwd(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return FA_OK;
}

}  // namespace

namespace fa {

int check_splitkv_args(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int Nq, int Nk, int d, const int* seqlens_k, float scale,
                       int dtype, int num_splits) {
  return check_forward(q, k, v, o, lse, B, H, Nq, Nk, d, dtype, scale, seqlens_k, num_splits,
                       nullptr, 0, false, false);
}

}  // namespace fa

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
           int N, int d, int causal, float scale, int dtype, fa_stream_t stream) {
  return run_forward(q, k, v, o, lse, B, H, N, N, d, causal, -1, -1, nullptr, scale, dtype, 1,
                     nullptr, 0, stream);
}

int fa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                  int H, int N, int d, int causal, int window_left, int window_right,
                  const int* seqlens_k, float scale, int dtype, fa_stream_t stream) {
  return run_forward(q, k, v, o, lse, B, H, N, N, d, causal, window_left, window_right,
                     seqlens_k, scale, dtype, 1, nullptr, 0, stream);
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int Nq, int d, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || d < 1 || num_splits <= 1) return 0;
  const uint64_t rows = (uint64_t)B * (uint64_t)H * (uint64_t)Nq * (uint64_t)num_splits;
  return (size_t)(rows * (uint64_t)d * 4 + rows * 4);
}

int fa_fwd_splitkv_num_splits(int B, int H, int Nq, int Nk, int num_sms) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || num_sms < 1) return 1;
  const long long units = (long long)B * H * ((Nq + 255) / 256);
  const long long kv_tiles = (Nk + 127) / 128;
  // Time model: waves of CTAs x (K/V tiles per part + a fixed cost of about 4 tiles per CTA
  // for its prologue, epilogue and share of the merge). Parts keep at least 2 tiles.
  const long long max_splits = std::max<long long>(1, std::min<long long>(fa::MAX_SPLITS,
                                                                          kv_tiles / 2));
  long long best = 1, best_cost = -1;
  for (long long s = 1; s <= max_splits; ++s) {
    const long long waves = (units * s + num_sms - 1) / num_sms;
    const long long cost = waves * ((kv_tiles + s - 1) / s + 4);
    if (best_cost < 0 || cost < best_cost) {
      best = s;
      best_cost = cost;
    }
  }
  return (int)best;
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int H, int Nq, int Nk, int d, int causal, int window_left, int window_right,
                   const int* seqlens_k, float scale, int dtype, int num_splits,
                   void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return run_forward(q, k, v, o, lse, B, H, Nq, Nk, d, causal, window_left, window_right,
                     seqlens_k, scale, dtype, num_splits, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

// Host-side checks of fa_bwd (nothing is enqueued).
int check_backward(const void* q, const void* k, const void* v, const void* o,
                   const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                   int H, int N, int d, float scale, int dtype, void* workspace,
                   size_t workspace_bytes, bool inputs_written = false,
                   const int* seqlens_k = nullptr) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace)
    return FA_ERR_NULL;
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return FA_ERR_SHAPE;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!isfinite(scale)) return FA_ERR_SCALE;
  const uint64_t bh = (uint64_t)B * (uint64_t)H;
  if (bh * (uint64_t)((N + 127) / 128) >= (1ull << 31)) return FA_ERR_SHAPE;
  const uint64_t elems = bh * (uint64_t)N * (uint64_t)d;
  if (elems > (1ull << 62) / 4) return FA_ERR_SHAPE;
  if (workspace_bytes < fa_bwd_workspace_size(B, H, N, d)) return FA_ERR_WORKSPACE;
  const uint64_t t_bytes = elems * 2, lse_bytes = bh * (uint64_t)N * 4;
  for (const void* p : {q, k, v, o, dout, static_cast<const void*>(dq),
                        static_cast<const void*>(dk), static_cast<const void*>(dv),
                        static_cast<const void*>(workspace)})
    if (reinterpret_cast<uintptr_t>(p) % 16) return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) % 4) return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(seqlens_k) % 4) return FA_ERR_ALIGN;
  struct Span { const void* p; uint64_t n; };
  const Span ins[] = {{q, t_bytes}, {k, t_bytes}, {v, t_bytes}, {o, t_bytes}, {dout, t_bytes},
                      {lse, lse_bytes}, {seqlens_k, seqlens_k ? (uint64_t)B * 4 : 0}};
  const Span outs[] = {{dq, t_bytes}, {dk, t_bytes}, {dv, t_bytes},
                       {workspace, fa_bwd_workspace_size(B, H, N, d)}};
  for (const Span& out : outs)
    for (const Span& in : ins)
      if (in.p && overlaps(out.p, out.n, in.p, in.n)) return FA_ERR_ALIAS;
  for (int i = 0; i < 4; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (overlaps(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return FA_ERR_ALIAS;
  if (inputs_written)   // as in check_forward
    for (int i = 0; i < 6; ++i)
      for (int j = i + 1; j < 6; ++j)
        if (overlaps(ins[i].p, ins[i].n, ins[j].p, ins[j].n)) return FA_ERR_ALIAS;
  int device = 0;
  const int rc = check_arch(&device);
  if (rc != FA_OK) return rc;
  return check_device_ptrs(device, {q, k, v, o, dout, lse, dq, dk, dv, workspace, seqlens_k});
}

}  // namespace

namespace {

// Streams on which the head groups' kernels of one host-buffer call run, in turn. A group's
// kernel cannot end before its longest CTA (a causal key walk over the whole sequence), so on
// one stream the groups' kernels form a chain of such walks; on several, one group's short
// CTAs fill the SMs while another's long ones finish. Measured at B=1, H=8, N=32768 (8
// groups): forward 2.14 -> 1.91 ms per call, backward 5.41 -> 4.89 ms, with three streams
// instead of one; no change at N=8192, where the copies dominate.
constexpr int kHostKernelStreams = 3;

// Per device: the two copy streams of fa_fwd_host / fa_bwd_host, the kernel streams and their
// events, created on first use and kept for the life of the process. One mutex serialises the
// enqueueing of the host-buffer calls, so that two callers never interleave their event
// records and waits.
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaStream_t kern[kHostKernelStreams] = {};
  std::vector<cudaEvent_t> events;
};
std::mutex g_host_mutex;
HostPipe g_host_pipe[kMaxDevices];

int host_pipe(int device, size_t events, HostPipe** out) {
  HostPipe& hp = g_host_pipe[device];
  if (!hp.in && cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) != cudaSuccess)
    return FA_ERR_CUDA;
  if (!hp.out && cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) != cudaSuccess)
    return FA_ERR_CUDA;
  for (cudaStream_t& k : hp.kern)
    if (!k && cudaStreamCreateWithFlags(&k, cudaStreamNonBlocking) != cudaSuccess)
      return FA_ERR_CUDA;
  while (hp.events.size() < events) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return FA_ERR_CUDA;
    hp.events.push_back(e);
  }
  *out = &hp;
  return FA_OK;
}

// Makes the copy and kernel streams of `hp` wait for the work already on `s` (recorded in
// `start`).
bool pipe_start(HostPipe* hp, cudaEvent_t start, cudaStream_t s) {
  if (cudaEventRecord(start, s) != cudaSuccess || cudaStreamWaitEvent(hp->in, start, 0) ||
      cudaStreamWaitEvent(hp->out, start, 0))
    return false;
  for (cudaStream_t k : hp->kern)
    if (cudaStreamWaitEvent(k, start, 0) != cudaSuccess) return false;
  return true;
}

constexpr int kMaxHostGroups = 8;   // head groups per host-buffer call, at most

// Number of head groups a host-buffer call is cut into (the groups' copies overlap the kernels
// of other groups, and the groups' kernels overlap one another on the kernel streams): as many
// as allowed, at most H and kMaxHostGroups, each with at least 16 MB of copies (below that, the
// per-group launch and copy set-up costs more than the overlap saves). Groups of equal size are
// preferred: the largest divisor of H within that bound, unless it is below half the bound.
// Measured on the backward at B=2, H=16, N=8192: 4 or 8 equal groups 2.53-2.55 ms per call,
// 5 or 6 unequal ones 2.88-2.94 ms.
int host_groups(int H, double copy_bytes) {
  const int most = (int)std::max<long long>(
      1, std::min<long long>({(long long)H, (long long)kMaxHostGroups,
                              (long long)(copy_bytes / (16.0 * (1 << 20)))}));
  int even = 1;
  for (int g = most; g >= 1; --g)
    if (H % g == 0) { even = g; break; }
  return 2 * even >= most ? even : most;
}

// Heads [h0, h0 + hc) of a [B, N, H, d] 16-bit array between host memory (pitch H * d) and a
// compact [B, N, hc, d] device array, as one pitched copy.
bool copy_heads(void* compact, void* host, bool to_device, int B, int N, int H, int h0, int hc,
                int d, cudaStream_t st) {
  const size_t row = (size_t)d * 2, width = (size_t)hc * row, pitch = (size_t)H * row;
  char* h = static_cast<char*>(host) + (size_t)h0 * row;
  return (to_device ? cudaMemcpy2DAsync(compact, width, h, pitch, width, (size_t)B * N,
                                        cudaMemcpyHostToDevice, st)
                    : cudaMemcpy2DAsync(h, pitch, compact, width, width, (size_t)B * N,
                                        cudaMemcpyDeviceToHost, st)) == cudaSuccess;
}

// The same for a [B, H, N] fp32 array (LSE): B blocks of hc * N floats.
bool copy_rows(float* compact, float* host, bool to_device, int B, int N, int H, int h0, int hc,
               cudaStream_t st) {
  const size_t width = (size_t)hc * N * 4, pitch = (size_t)H * N * 4;
  float* h = host + (size_t)h0 * N;
  return (to_device ? cudaMemcpy2DAsync(compact, width, h, pitch, width, (size_t)B,
                                        cudaMemcpyHostToDevice, st)
                    : cudaMemcpy2DAsync(h, pitch, compact, width, width, (size_t)B,
                                        cudaMemcpyDeviceToHost, st)) == cudaSuccess;
}

}  // namespace

extern "C" {

int fa_fwd_host_masked(const void* q_h, const void* k_h, const void* v_h, void* o_h,
                       float* lse_h, void* q_d, void* k_d, void* v_d, void* o_d, float* lse_d,
                       int B, int H, int N, int d, int causal, int window_left,
                       int window_right, const int* seqlens_k, float scale, int dtype,
                       fa_stream_t stream) {
  if (!q_h || !k_h || !v_h || !o_h || !lse_h) return FA_ERR_NULL;
  int rc = check_forward(q_d, k_d, v_d, o_d, lse_d, B, H, N, N, d, dtype, scale, seqlens_k, 1,
                         nullptr, 0, true);
  if (rc != FA_OK) return rc;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return FA_ERR_CUDA;
  const int groups = host_groups(H, 4.0 * B * H * (double)N * d * 2 + (double)B * H * N * 4);
  std::lock_guard<std::mutex> lock(g_host_mutex);
  HostPipe* hp = nullptr;
  rc = host_pipe(device, 2 + 2 * (size_t)groups, &hp);
  if (rc != FA_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaEvent_t* ev = hp->events.data();   // [0] start, [1] end, then in/kernel per group
  // The copy and kernel streams start after the work already on `stream`.
  if (!pipe_start(hp, ev[0], s)) return FA_ERR_CUDA;
  // Group g: heads [h0, h1) of every batch, packed into a compact [B, N, h1 - h0, d] problem
  // at the next free offset of the device buffers.
  size_t packed = 0, packed_lse = 0;   // bytes / floats used so far
  for (int g = 0; g < groups; ++g) {
    const int h0 = (int)((int64_t)H * g / groups), h1 = (int)((int64_t)H * (g + 1) / groups);
    const int hc = h1 - h0;
    char* qd = static_cast<char*>(q_d) + packed;
    char* kd = static_cast<char*>(k_d) + packed;
    char* vd = static_cast<char*>(v_d) + packed;
    char* od = static_cast<char*>(o_d) + packed;
    float* ld = lse_d + packed_lse;
    cudaStream_t ks = hp->kern[g % kHostKernelStreams];
    if (!copy_heads(qd, const_cast<void*>(q_h), true, B, N, H, h0, hc, d, hp->in) ||
        !copy_heads(kd, const_cast<void*>(k_h), true, B, N, H, h0, hc, d, hp->in) ||
        !copy_heads(vd, const_cast<void*>(v_h), true, B, N, H, h0, hc, d, hp->in) ||
        cudaEventRecord(ev[2 + 2 * g], hp->in) != cudaSuccess ||
        cudaStreamWaitEvent(ks, ev[2 + 2 * g], 0) != cudaSuccess)
      return FA_ERR_CUDA;
    // groups span every batch, so the per-batch key lengths apply to each group unchanged
    rc = run_forward(qd, kd, vd, od, ld, B, hc, N, N, d, causal, window_left, window_right,
                     seqlens_k, scale, dtype, 1, nullptr, 0,
                     reinterpret_cast<fa_stream_t>(ks));
    if (rc != FA_OK) return rc;
    if (cudaEventRecord(ev[3 + 2 * g], ks) != cudaSuccess ||
        cudaStreamWaitEvent(hp->out, ev[3 + 2 * g], 0) != cudaSuccess ||
        !copy_heads(od, o_h, false, B, N, H, h0, hc, d, hp->out) ||
        !copy_rows(ld, lse_h, false, B, N, H, h0, hc, hp->out))
      return FA_ERR_CUDA;
    packed += (size_t)B * N * hc * d * 2;
    packed_lse += (size_t)B * hc * N;
  }
  // `stream` reaches this point once the last output copy is done (the output stream has
  // waited for every group's kernel).
  if (cudaEventRecord(ev[1], hp->out) != cudaSuccess || cudaStreamWaitEvent(s, ev[1], 0))
    return FA_ERR_CUDA;
  return FA_OK;
}

int fa_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                void* q_d, void* k_d, void* v_d, void* o_d, float* lse_d, int B, int H, int N,
                int d, int causal, float scale, int dtype, fa_stream_t stream) {
  return fa_fwd_host_masked(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d, B, H, N, d,
                            causal, -1, -1, nullptr, scale, dtype, stream);
}

int fa_bwd_host_masked(const void* q_h, const void* k_h, const void* v_h, const void* o_h,
                       const void* do_h, const float* lse_h, void* dq_h, void* dk_h, void* dv_h,
                       void* q_d, void* k_d, void* v_d, void* o_d, void* do_d, float* lse_d,
                       void* dq_d, void* dk_d, void* dv_d, void* workspace,
                       size_t workspace_bytes, int B, int H, int N, int d, int causal,
                       int window_left, int window_right, const int* seqlens_k, float scale,
                       int dtype, fa_stream_t stream) {
  if (!q_h || !k_h || !v_h || !o_h || !do_h || !lse_h || !dq_h || !dk_h || !dv_h)
    return FA_ERR_NULL;
  int rc = check_backward(q_d, k_d, v_d, o_d, do_d, lse_d, dq_d, dk_d, dv_d, B, H, N, d, scale,
                          dtype, workspace, workspace_bytes, true, seqlens_k);
  if (rc != FA_OK) return rc;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return FA_ERR_CUDA;
  const int groups = host_groups(H, 8.0 * B * H * (double)N * d * 2 + (double)B * H * N * 4);
  std::lock_guard<std::mutex> lock(g_host_mutex);
  HostPipe* hp = nullptr;
  rc = host_pipe(device, 2 + 2 * (size_t)groups, &hp);
  if (rc != FA_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaEvent_t* ev = hp->events.data();
  if (!pipe_start(hp, ev[0], s)) return FA_ERR_CUDA;
  // Each group's three kernels get a workspace of their own, at a 16-byte aligned offset, when
  // those fit in the caller's workspace (the groups' sizes add up to the whole problem's, plus
  // the padding); otherwise every group runs on one kernel stream, after the previous group,
  // at the start of the workspace.
  size_t ws_total = 0;
  for (int g = 0; g < groups; ++g) {
    const int hc = (int)((int64_t)H * (g + 1) / groups) - (int)((int64_t)H * g / groups);
    ws_total += (fa_bwd_workspace_size(B, hc, N, d) + 15) / 16 * 16;
  }
  const int kstreams = ws_total <= workspace_bytes ? kHostKernelStreams : 1;
  size_t packed = 0, packed_lse = 0, ws_off = 0;
  for (int g = 0; g < groups; ++g) {
    const int h0 = (int)((int64_t)H * g / groups), h1 = (int)((int64_t)H * (g + 1) / groups);
    const int hc = h1 - h0;
    cudaStream_t ks = hp->kern[g % kstreams];
    const size_t ws_g = kstreams > 1 ? fa_bwd_workspace_size(B, hc, N, d) : workspace_bytes;
    void* ws = static_cast<char*>(workspace) + (kstreams > 1 ? ws_off : 0);
    ws_off += (ws_g + 15) / 16 * 16;
    char* dev[8];
    void* bases[8] = {q_d, k_d, v_d, o_d, do_d, dq_d, dk_d, dv_d};
    for (int t = 0; t < 8; ++t) dev[t] = static_cast<char*>(bases[t]) + packed;
    float* ld = lse_d + packed_lse;
    const void* ins[5] = {q_h, k_h, v_h, o_h, do_h};
    bool ok = true;
    for (int t = 0; t < 5 && ok; ++t)
      ok = copy_heads(dev[t], const_cast<void*>(ins[t]), true, B, N, H, h0, hc, d, hp->in);
    if (!ok || !copy_rows(ld, const_cast<float*>(lse_h), true, B, N, H, h0, hc, hp->in) ||
        cudaEventRecord(ev[2 + 2 * g], hp->in) != cudaSuccess ||
        cudaStreamWaitEvent(ks, ev[2 + 2 * g], 0) != cudaSuccess)
      return FA_ERR_CUDA;
    rc = fa_bwd_masked(dev[0], dev[1], dev[2], dev[3], dev[4], ld, dev[5], dev[6], dev[7], B, hc,
                       N, d, causal, window_left, window_right, seqlens_k, scale, dtype, ws,
                       ws_g, reinterpret_cast<fa_stream_t>(ks));
    if (rc != FA_OK) return rc;
    void* outs[3] = {dq_h, dk_h, dv_h};
    if (cudaEventRecord(ev[3 + 2 * g], ks) != cudaSuccess ||
        cudaStreamWaitEvent(hp->out, ev[3 + 2 * g], 0) != cudaSuccess)
      return FA_ERR_CUDA;
    for (int t = 0; t < 3; ++t)
      if (!copy_heads(dev[5 + t], outs[t], false, B, N, H, h0, hc, d, hp->out))
        return FA_ERR_CUDA;
    packed += (size_t)B * N * hc * d * 2;
    packed_lse += (size_t)B * hc * N;
  }
  if (cudaEventRecord(ev[1], hp->out) != cudaSuccess || cudaStreamWaitEvent(s, ev[1], 0))
    return FA_ERR_CUDA;
  return FA_OK;
}

int fa_bwd_host(const void* q_h, const void* k_h, const void* v_h, const void* o_h,
                const void* do_h, const float* lse_h, void* dq_h, void* dk_h, void* dv_h,
                void* q_d, void* k_d, void* v_d, void* o_d, void* do_d, float* lse_d,
                void* dq_d, void* dk_d, void* dv_d, void* workspace, size_t workspace_bytes,
                int B, int H, int N, int d, int causal, float scale, int dtype,
                fa_stream_t stream) {
  return fa_bwd_host_masked(q_h, k_h, v_h, o_h, do_h, lse_h, dq_h, dk_h, dv_h, q_d, k_d, v_d,
                            o_d, do_d, lse_d, dq_d, dk_d, dv_d, workspace, workspace_bytes, B,
                            H, N, d, causal, -1, -1, nullptr, scale, dtype, stream);
}

int fa_selftest_wait_timeout(int limit_us, fa_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return FA_ERR_SHAPE;
  int device = 0;
  const int rc = check_arch(&device);
  if (rc != FA_OK) return rc;
  if (fa::launch_selftest_wait(1000ull * (unsigned long long)limit_us,
                               reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return FA_OK;
}

int fa_get_device_error(fa_stream_t stream) {
  int value = 0, bwd_value = 0;
  if (fa::read_and_clear_device_error(reinterpret_cast<cudaStream_t>(stream), &value) !=
          cudaSuccess ||
      fa::read_and_clear_bwd_error(&bwd_value) != cudaSuccess)
    return FA_ERR_CUDA;
  return (value == 0 && bwd_value == 0) ? FA_OK : FA_ERR_TIMEOUT;
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  const uint64_t rows = (uint64_t)B * (uint64_t)H * (uint64_t)N;
  return (size_t)(rows * (uint64_t)d * 4 + rows * 4);
}

}  // extern "C"

extern "C" {

int fa_bwd_masked(const void* q, const void* k, const void* v, const void* o,
                  const void* dout, const float* lse, void* dq, void* dk, void* dv, int B, int H,
                  int N, int d, int causal, int window_left, int window_right,
                  const int* seqlens_k, float scale, int dtype, void* workspace,
                  size_t workspace_bytes, fa_stream_t stream) {
  const int rc = check_backward(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, dtype,
                                workspace, workspace_bytes, false, seqlens_k);
  if (rc != FA_OK) return rc;
  const uint64_t elems = (uint64_t)B * (uint64_t)H * (uint64_t)N * (uint64_t)d;
  fa::BwdParams p;
  const bool fp16 = dtype == FA_FP16;
  if (!encode_bnhd(&p.tm_q, q, B, H, N, d, fp16) || !encode_bnhd(&p.tm_k, k, B, H, N, d, fp16) ||
      !encode_bnhd(&p.tm_v, v, B, H, N, d, fp16) ||
      !encode_bnhd(&p.tm_do, dout, B, H, N, d, fp16))
    return FA_ERR_CUDA;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.dq_acc = static_cast<float*>(workspace);
  p.dpre = static_cast<float*>(workspace) + elems;
  p.B = B;
  p.H = H;
  p.N = N;
  p.d = d;
  p.causal = causal ? 1 : 0;
  // a bound wider than the sequence is no narrower than none, and keeps the kernel's index
  // arithmetic within int
  p.window_left = window_left < 0 ? -1 : std::min(window_left, N);
  p.window_right = window_right < 0 ? -1 : std::min(window_right, N);
  p.seqlens_k = seqlens_k;
  p.fp16 = fp16 ? 1 : 0;
  p.scale = scale;
  if (fa::launch_bwd(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return FA_OK;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
           int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
           fa_stream_t stream) {
  return fa_bwd_masked(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, -1, -1, nullptr,
                       scale, dtype, workspace, workspace_bytes, stream);
}

}  // extern "C"
