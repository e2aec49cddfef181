// fa_noalloc.cu -- fa_fwd_splitkv_noalloc: the split-K/V forward with a workspace that lives
// inside the library, for callers that cannot allocate device memory when they call.
//
// Who needs it: code that runs inside a host which owns the whole device-memory budget (a
// plugin of a serving engine or framework that forbids allocations after start-up), and
// latency-critical loops where an allocation, with the device synchronisation cudaMalloc may
// imply, is not acceptable. Such callers still pass their own inputs and outputs; only the
// scratch space for the K/V parts comes from here.
//
// The scratch is one file-scope device array, kNoAllocScratchBytes (8 MiB) large. Every GPU
// that loads this library keeps it for the life of the process. All calls on a device share
// it and it keeps the last call's contents; nothing in it has to start at zero, because the
// attention kernel writes every part row (O and LSE) of the parts a call uses before the merge
// kernel reads them. Calls whose work overlaps on the GPU (different streams, no ordering
// between them) race on the array; order them on one stream or with events.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

// Host code must not use this name as a device address: on the host it only identifies the
// symbol. Its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};   // id of the context the address is from

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the current CUDA context (0 when it cannot be read). A device reset destroys
// the primary context; the next one gets a new id, and the library's module (with this
// array) is loaded again at a possibly different address.
unsigned long long current_context_id() {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_noalloc_scratch on the current device, looked up with that device
// current the first time it is needed in its context (again after a device reset). Returns
// FA_OK or FA_ERR_CUDA; a failed lookup leaves no CUDA error behind for the caller.
int scratch_for_current_device(void** out) {
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  const unsigned long long ctx = current_context_id();
  if (ctx == 0) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[device] || g_scratch_ctx[device] != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      g_scratch_ptr[device] = nullptr;
      return FA_ERR_CUDA;
    }
    g_scratch_ptr[device] = ptr;
    g_scratch_ctx[device] = ctx;
  }
  *out = g_scratch_ptr[device];
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int Nq, int Nk, int d, int causal, int window_left,
                           int window_right, const int* seqlens_k, float scale, int dtype,
                           int num_splits, fa_stream_t stream) {
  // The checks fa_fwd_splitkv makes on everything but the workspace come first, so that these
  // arguments give the same codes as there; then the size check against the built-in buffer.
  int rc = fa::check_splitkv_args(q, k, v, o, lse, B, H, Nq, Nk, d, seqlens_k, scale, dtype,
                                  num_splits);
  if (rc != FA_OK) return rc;
  const size_t need = fa_fwd_splitkv_workspace_size(B, H, Nq, d, num_splits);
  if (need > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  rc = scratch_for_current_device(&scratch);
  if (rc != FA_OK) return rc;
  return fa_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, causal, window_left, window_right,
                        seqlens_k, scale, dtype, num_splits, scratch, kNoAllocScratchBytes,
                        stream);
}

}  // extern "C"
