// pre_attn_run_noalloc: the decode step for callers that cannot allocate
// device memory.
//
// pre_attn_run() wants a caller-provided workspace.  Some callers have no way
// to produce one: a plugin loaded into a host runtime that owns all device
// memory through its own pool and hands out none, or a process whose device
// memory is capped so that any cudaMalloc after start-up fails.  This entry
// point runs the same prologue and skinny-GEMV kernels as pre_attn_run, with
// the kernels' scratch (the status word and the quantised activations with
// their scales) in a fixed array that lives in this file.  It allocates nothing: no cudaMalloc, no cudaFree, no
// allocating library call.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/pre_attn.h"

namespace {

// The static scratch: every GPU that loads this library holds it until the
// process exits.  Zero-initialised at module load.
constexpr size_t kScratchBytes = (size_t)2 << 20;  // 2 MiB
__device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

// Host code may not use g_noalloc_scratch as a device address (it is a host
// stand-in); its device address is looked up once per device.
constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// The scratch's device address on the current device, looked up (with that
// device current) on the first call made on it.
int scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" {

int pre_attn_run_noalloc(pa_handle *h, int M, const pa_step_inputs *in, const pa_weights *wt,
                         const pa_caches *caches, const pa_outputs *out, void *stream) {
  if (!h) return PA_ERR_NULL;
  if (M < 0 || M > 16) return PA_ERR_SHAPE;  // the skinny (decode) path only
  const size_t need = pre_attn_workspace_bytes(h, M);
  if (need == 0 || need > kScratchBytes) return PA_ERR_SHAPE;  // beyond max_tokens or the 2 MiB scratch
  if (M == 0) return PA_OK;
  void *scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != PA_OK) return st;
  // Every call reuses the array and finds the previous call's contents; the
  // part this call uses is cleared first (the status word must start at zero).
  if (cudaMemsetAsync(scratch, 0, need, (cudaStream_t)stream) != cudaSuccess) return PA_ERR_CUDA;
  return pre_attn_run(h, M, in, wt, caches, out, scratch, kScratchBytes, stream);
}

}  // extern "C"
