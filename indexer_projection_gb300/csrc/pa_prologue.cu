// Prologue of the pre-attention step: one CTA per token row.
// residual add, Gemma RMSNorm and the activation quantiser (pa_norm.cuh),
// used ahead of the tensor-core path and of the skinny path at large H.
// HBM-bound: 16-byte coalesced loads and stores, the row held in registers,
// warp-shuffle + shared-memory block reductions for sum(acc^2) and amax.
#include "pa_device.cuh"
#include "pa_launch.h"
#include "pa_norm.cuh"

namespace pa {

// NTHR threads a row, MAXC chunks of 8 elements per thread: H <= 8 * NTHR *
// MAXC.  The row stays in registers, so MAXC is sized to H.  Many rows (the
// tensor-core path): 256 threads a row, more rows resident per SM.  A few
// rows (the skinny path, which waits on this kernel): 1024 threads a row, so
// the per-element work of the correctly rounded norm is spread 4x wider and
// the row is done sooner.
template <int WFMT, int NTHR, int MAXC>
__global__ void __launch_bounds__(NTHR) prologue_kernel(Params p, int use_pdl) {
  __shared__ float red[NTHR / 32];
  __shared__ float2 red2[NTHR / 32];
  if (use_pdl) {
    pdl_trigger();
    pdl_wait();
  }
  const int m = blockIdx.x;
  const int ksf = p.H >> 5;
  if (m >= p.M) {  // MXFP8 padding rows of the tensor-core path: scale 1, codes unused
    if (WFMT == 1)
      for (int kb = threadIdx.x; kb < ksf; kb += NTHR) p.xsf[sf128x4_offset(m, kb, ksf)] = 127;
    return;
  }
  norm_quant_row<WFMT, NTHR, MAXC>(p, m, red, red2);
}

__global__ void pack_scales_kernel(const uint8_t *src, uint8_t *dst, int rows, int ksf) {
  const int64_t rpad = ((int64_t)rows + 127) / 128 * 128;
  const int64_t total = rpad * ksf;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / ksf;
    const int kb = (int)(i - r * ksf);
    dst[sf128x4_offset(r, kb, ksf)] = r < rows ? src[i] : (uint8_t)127;
  }
}

namespace {
// H <= 16384: 1024 threads need at most 2 chunks, 256 threads at most 8
cudaError_t launch_1024(const Params &p, cudaLaunchConfig_t &cfg, bool pdl) {
  cfg.blockDim = dim3(1024);
  const bool mx = p.weight_fmt == 1;
  if (mx) return cudaLaunchKernelEx(&cfg, prologue_kernel<1, 1024, 2>, p, (int)pdl);  // (one chunk spills)
  if (p.H <= 8 * 1024) return cudaLaunchKernelEx(&cfg, prologue_kernel<0, 1024, 1>, p, (int)pdl);
  return cudaLaunchKernelEx(&cfg, prologue_kernel<0, 1024, 2>, p, (int)pdl);
}
cudaError_t launch_256(const Params &p, cudaLaunchConfig_t &cfg, bool pdl) {
  cfg.blockDim = dim3(256);
  const int maxc = (p.H + 8 * 256 - 1) / (8 * 256);
  const bool mx = p.weight_fmt == 1;
  if (maxc <= 2) return cudaLaunchKernelEx(&cfg, mx ? prologue_kernel<1, 256, 2> : prologue_kernel<0, 256, 2>, p, (int)pdl);
  if (maxc <= 3) return cudaLaunchKernelEx(&cfg, mx ? prologue_kernel<1, 256, 3> : prologue_kernel<0, 256, 3>, p, (int)pdl);
  if (maxc <= 4) return cudaLaunchKernelEx(&cfg, mx ? prologue_kernel<1, 256, 4> : prologue_kernel<0, 256, 4>, p, (int)pdl);
  return cudaLaunchKernelEx(&cfg, mx ? prologue_kernel<1, 256, 8> : prologue_kernel<0, 256, 8>, p, (int)pdl);
}
}  // namespace

cudaError_t launch_prologue(const Params &p, int grid, bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(grid);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  // fewer rows than a fraction of the SMs: the row latency is the step's
  return grid <= 64 ? launch_1024(p, cfg, pdl) : launch_256(p, cfg, pdl);
}

cudaError_t launch_pack_scales(const uint8_t *src, uint8_t *dst, int rows, int ksf, cudaStream_t stream) {
  const int64_t total = ((int64_t)rows + 127) / 128 * 128 * ksf;
  const int grid = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, pack_scales_kernel, src, dst, rows, ksf);
}

}  // namespace pa
