// pre_attn_run_noalloc: the step for callers that cannot allocate device
// memory, and pre_attn_noalloc_status, its status reader.
//
// pre_attn_run() wants a caller-provided workspace.  Some callers have no way
// to produce one: a plugin loaded into a host runtime that owns all device
// memory through its own pool and hands out none, or a process whose device
// memory is capped so that any cudaMalloc after start-up fails.  This entry
// point runs the same kernels as pre_attn_run for up to 16 token rows, with
// the kernels' scratch (the status word and the quantised activations with
// their scales) in a fixed array that lives in this file.  It allocates
// nothing: no cudaMalloc, no cudaFree, no allocating library call.
#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pre_attn.h"
#include "pa_launch.h"

namespace {

// The static scratch: every GPU that loads this library holds it until the
// process exits.  Zero-initialised at module load.
constexpr size_t kScratchBytes = (size_t)2 << 20;  // 2 MiB
constexpr int kMaxRows = 16;
__device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

// In host code g_noalloc_scratch names a host-side stand-in, not the device
// array: its device address is looked up with cudaGetSymbolAddress, with the
// device current, and kept per device together with the id of the context
// it belongs to.  A later call on another context of that device (after
// cudaDeviceReset, say) looks the address up again; calls on the same
// context read the cache without a lock.
constexpr int kMaxDevices = 64;
struct ScratchEntry {
  std::atomic<unsigned long long> ctx_id{0};  // 0: nothing cached
  std::atomic<void *> ptr{nullptr};
};
ScratchEntry g_scratch[kMaxDevices];
std::mutex g_lookup_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <typename F>
F driver_fn(const char *name) {
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(fn);
}

// The id of the context current on this thread (0 if none is).
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// The scratch's device address on the current device and context.
int scratch_for_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pa::record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  ScratchEntry &en = g_scratch[dev];
  const unsigned long long id = current_ctx_id();
  if (id != 0 && en.ctx_id.load(std::memory_order_acquire) == id) {
    *out = en.ptr.load(std::memory_order_relaxed);
    return PA_OK;
  }
  std::lock_guard<std::mutex> lock(g_lookup_mu);
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // also makes the device's context current
  if (e != cudaSuccess) return pa::record_cuda_error(e);
  if (!p) return PA_ERR_CUDA;
  en.ptr.store(p, std::memory_order_relaxed);
  en.ctx_id.store(current_ctx_id(), std::memory_order_release);
  *out = p;
  return PA_OK;
}

}  // namespace

extern "C" {

int pre_attn_run_noalloc(pa_handle *h, int M, const pa_step_inputs *in, const pa_weights *wt,
                         const pa_caches *caches, const pa_outputs *out, void *stream) {
  if (!h) return PA_ERR_NULL;
  if (M < 0 || M > kMaxRows) return PA_ERR_SHAPE;  // up to 16 rows, on whichever path the handle selects
  const size_t need = pre_attn_workspace_bytes(h, M);
  if (need == 0 || need > kScratchBytes) return PA_ERR_SHAPE;  // beyond max_tokens or the 2 MiB scratch
  if (M == 0) return PA_OK;
  void *scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != PA_OK) return st;
  // Every call reuses the array and finds the previous call's contents; the
  // part this call uses is cleared first (the status word must start at zero).
  const cudaError_t e = cudaMemsetAsync(scratch, 0, need, (cudaStream_t)stream);
  if (e != cudaSuccess) return pa::record_cuda_error(e);
  return pre_attn_run(h, M, in, wt, caches, out, scratch, kScratchBytes, stream);
}

int pre_attn_noalloc_status(uint32_t *flags, void *stream) {
  if (!flags) return PA_ERR_NULL;
  void *scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != PA_OK) return st;
  // the status word sits at the start of the scratch, as in a workspace
  return pre_attn_device_status(scratch, flags, stream);
}

}  // extern "C"
