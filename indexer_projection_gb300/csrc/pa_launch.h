// Host-side launchers of the pre-attention kernels (one per translation unit).
#pragma once

#include <cuda_runtime.h>

namespace pa {

struct Params;

// Keep `e` as this thread's pre_attn_last_cuda_error() text; returns PA_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// Raise a kernel's dynamic shared-memory limit once per (kernel, device),
// kept out of the per-call path so the launch sequence also works inside
// stream capture.  Keyed on the kernel's address: template instances share
// one C++ type.
inline cudaError_t ensure_smem_attr(const void *kern, int bytes) {
  struct Entry {
    const void *k;
    int dev, bytes;
  };
  static Entry table[64];
  static int n = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n; ++i)
    if (table[i].k == kern && table[i].dev == dev && table[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && n < 64) table[n++] = Entry{kern, dev, bytes};
  return e;
}

// SM count of the current device (cached per device); -1 if the query fails.
inline int current_device_sms() {
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (sms[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    sms[dev] = n;
  }
  return sms[dev];
}

// Prologue over `grid` CTAs (M rows, plus padding rows of the MXFP8 scale grid).
// A grid of at most early_max CTAs triggers the next kernel's launch at its
// start, a larger one after its rows' work.
cudaError_t launch_prologue(const Params &p, int grid, bool pdl, int early_max, cudaStream_t stream);
// CTAs an SM holds of the prologue kernel launch_prologue picks for H, the
// weight format and the grid width (wide: grid <= 64, 1024 threads a CTA).
cudaError_t prologue_ctas_per_sm(int H, int weight_fmt, bool wide, int *per_sm);
// Prologue of the skinny path: one thread-block cluster per row (M <= 16).
cudaError_t launch_prologue_rows(const Params &p, bool pdl, cudaStream_t stream);
// Row-major [rows, ksf] E8M0 -> F8_128x4 layout.
cudaError_t launch_pack_scales(const uint8_t *src, uint8_t *dst, int rows, int ksf, cudaStream_t stream);

// Skinny-M path (M <= 16): FP8 GEMV on one thread-block cluster per head,
// the head epilogue fused behind the in-cluster reduction.  With `fused`
// (allowed when gemv_fuses_prologue(H, weight format)) the kernel also does
// the prologue's work and no prologue is launched.
bool gemv_fuses_prologue(int H, int weight_fmt);
cudaError_t launch_gemv(const Params &p, bool fused, bool pdl, cudaStream_t stream);
// Resident clusters of 16 of that kernel at hidden size H (0: clusters of 16
// cannot be co-scheduled).
int gemv_regular_clusters(int weight_fmt, int H);
// The persistent variant for many heads (pa_gemv_persist.cu): the clusters
// to launch, or 0 where it is not used (H > 6144, not launchable, or -
// unless forced - the regular grid fits one wave).
int gemv_persist_clusters(int n_heads, int H, int weight_fmt, bool force);
cudaError_t launch_gemv_persist(const Params &p, int clusters, bool pdl, cudaStream_t stream);

// Tensor-core path: persistent tcgen05 GEMM with the fused head epilogue,
// on single CTAs (128 x 128 tiles) or on CTA pairs (cta_group::2, 256 x 256).
cudaError_t launch_gemm(const Params &p, int num_sms, int grid_override, bool pdl, cudaStream_t stream);
cudaError_t launch_gemm_pair(const Params &p, int num_sms, int64_t l2_bytes, int grid_override, bool pdl,
                             cudaStream_t stream);

}  // namespace pa
