// Signal mode, the consumer side: a kernel that waits until the done words
// a pre-attention step publishes (pa_outputs.done) reach the step's epoch
// ("vllm.models.minimax_m3.amd.mono.kernels.pre_attn", emit_k1: the indexer
// scorers poll the head tasks' done flags before they read the new keys).
//
// Every wait is bounded: a word that has not reached the epoch when the
// limit runs out raises PA_DEV_WAIT_TIMEOUT in the caller's status word and
// the thread gives up; the kernel always returns.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/pre_attn.h"
#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

constexpr int kWaitThreads = 128;

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Thread i waits for words i, i + stride, ...; the limit is counted from the
// thread's first poll, so a late-scheduled CTA still gets the whole limit.
__global__ void __launch_bounds__(kWaitThreads) pa_wait_done_kernel(const uint32_t *done, int64_t count,
                                                                     uint32_t epoch, uint64_t limit_ns,
                                                                     uint32_t *status) {
  const int64_t stride = (int64_t)gridDim.x * kWaitThreads;
  const uint64_t t0 = globaltimer();
  for (int64_t i = (int64_t)blockIdx.x * kWaitThreads + threadIdx.x; i < count; i += stride) {
    while (ld_acquire_u32(done + i) != epoch) {
      if (globaltimer() - t0 > limit_ns) {
        set_status(status, kDevWaitTimeout);
        return;
      }
      __nanosleep(64);
    }
  }
}

}  // namespace pa

extern "C" int pre_attn_wait_done(const uint32_t *done, int64_t count, uint32_t epoch, uint32_t timeout_us,
                                  uint32_t *status, void *stream) {
  if (!done || !status) return PA_ERR_NULL;
  if (count < 1) return PA_ERR_SHAPE;
  if (epoch == 0 || timeout_us < 1 || timeout_us > 10000000u) return PA_ERR_CONFIG;
  if (reinterpret_cast<uintptr_t>(done) % 4 || reinterpret_cast<uintptr_t>(status) % 4) return PA_ERR_ALIGN;
  const int64_t blocks = (count + pa::kWaitThreads - 1) / pa::kWaitThreads;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)(blocks < 1024 ? blocks : 1024));
  cfg.blockDim = dim3(pa::kWaitThreads);
  cfg.stream = (cudaStream_t)stream;
  // may start while the step's last kernel runs: it follows the words, not
  // the kernel's completion
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, pa::pa_wait_done_kernel, done, count, epoch, (uint64_t)timeout_us * 1000ull, status);
  return e == cudaSuccess ? PA_OK : pa::record_cuda_error(e);
}
