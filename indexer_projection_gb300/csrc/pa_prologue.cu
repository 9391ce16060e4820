// Prologue of the pre-attention step: residual add, Gemma RMSNorm and the
// activation quantiser (pa_norm.cuh).
//   pa_prologue_kernel       one CTA per token row: the tensor-core path's many
//                         rows (HBM-bound: 16-byte coalesced loads and stores,
//                         the row in registers, block reductions)
//   pa_prologue_rows_kernel  one thread-block cluster per token row, a K slice
//                         per CTA: the skinny path's few rows, whose latency
//                         the step waits on; the correctly rounded norm costs
//                         ~30 instructions an element, too much for a few
//                         SMs, so each row is spread over 8 SMs and the row
//                         sums are exchanged through distributed shared memory
//                         (one exchange carries the sum of squares and the
//                         per-channel amax)
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
// The tensor-core kernel that follows is launched when every CTA of this
// grid has passed its trigger, and it takes a whole SM's registers and
// shared memory for its CTA.  A grid of more than one wave triggers after
// the row's work (use_pdl 1), so the GEMM's CTAs do not take SMs this grid's
// later rows still need (a trigger at the start let them do that and
// stretched a two-wave 448-row prologue fourfold).  A grid resident all at
// once with at most two CTAs an SM triggers at its start (use_pdl 2): the
// GEMM's CTAs then take each SM as its rows finish and set up while the rest
// run (measured: 256 rows 35.6 -> 34.3 us a step; at 448 rows, three CTAs on
// most SMs, the early trigger was slower, 33.2 against 32.7 us).
template <int WFMT, int NTHR, int MAXC>
__global__ void __launch_bounds__(NTHR) pa_prologue_kernel(Params p, int use_pdl) {
  __shared__ float2 red2[NTHR / 32];
  if (use_pdl) pdl_wait();
  if (use_pdl == 2) pdl_trigger();
  const int m = blockIdx.x;
  const int ksf = p.H >> 5;
  if (m >= p.M) {  // MXFP8 padding rows of the tensor-core path: scale 1, codes unused
    if (WFMT == 1)
      for (int kb = threadIdx.x; kb < ksf; kb += NTHR) p.xsf[sf128x4_offset(m, kb, ksf)] = 127;
  } else {
    norm_quant_row<WFMT, NTHR, MAXC>(p, m, red2);
  }
  if (use_pdl == 1) pdl_trigger();
}

// One cluster of C CTAs per token row (blockIdx.x / C); CTA r takes the
// row's elements [r * kc, (r + 1) * kc), kc a multiple of 32 (one 8-element
// chunk a thread; the four chunks of an MXFP8 block in lanes 4i .. 4i + 3).
// Each CTA sends its double-float partial sum of acc^2, and for the
// per-channel format its partial maximum of |acc * (1 + gam)| (absprod_max8),
// to every CTA of the cluster in one byte-counted st.async; each CTA combines
// the C partials in the same order, so all agree bit for bit on rstd and on
// the scale, and one exchange serves both.
// The row's inputs are prefetched into L2 before the wait on the producing
// kernel (a hint: the loads after the wait still see its writes); after the
// wait CTA 0 of the row prefetches the row's cos / sin line for the GEMV's
// head epilogue.
template <int WFMT, int C, int NT = 128 * 16 / C>
__global__ void __launch_bounds__(NT) pa_prologue_rows_kernel(Params p, int kc, int use_pdl) {
  constexpr int NTHR = NT;
  constexpr int W = NTHR / 32;
  constexpr int XB = WFMT == 0 ? 16 : 8;  // bytes a CTA sends to each CTA
  __shared__ float4 ex1[C];               // the C partials: sum of acc^2 (hi, lo), max product (hi, lo)
  __shared__ float4 wred[W];
  __shared__ __align__(8) uint64_t bar1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m = blockIdx.x / C, r = (int)cta_rank();
  const int H = p.H, ksf = H >> 5;
  const int k0 = r * kc, k1 = k0 + kc < H ? k0 + kc : H;
  const int c = (k0 >> 3) + tid;  // this thread's chunk of the row
  const bool act = k0 + 8 * tid < k1;
  if (tid == 0) {
    mbar_init(&bar1, 1);
    mbar_expect_tx(&bar1, C * XB);
    fence_mbar_init();
  }
  cluster_arrive_relaxed();
  const uint4 *ar = reinterpret_cast<const uint4 *>(p.ar + (int64_t)m * H) + c;
  const uint4 *res = reinterpret_cast<const uint4 *>(p.res + (int64_t)m * H) + c;
  const bool cs_thread = r == 0 && tid == 0;
  uint4 gw = make_uint4(0u, 0u, 0u, 0u);
  if (act) {
    gw = __ldg(reinterpret_cast<const uint4 *>(p.g_in) + c);  // a model constant
    prefetch_l2(ar);
    prefetch_l2(res);
  }
  if (cs_thread) prefetch_l2(p.pos + m);
  if (use_pdl) {
    pdl_trigger();
    pdl_wait();
  }
  int64_t cpos = -1;  // loaded now, used last
  if (cs_thread) cpos = ld_i64(p.pos + m);
  float acc[8];
  float sh = 0.f, sl = 0.f, mh = 0.f, ml = 0.f;
  if (act) {
    uint4 rb;
    acc8(__ldcs(ar), __ldcs(res), acc, rb, sh, sl);
    if (p.residual) __stcs(reinterpret_cast<uint4 *>(p.residual + (int64_t)m * H) + c, rb);
    if (WFMT == 0) absprod_max8(acc, gw, mh, ml);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, sh, o), ol = __shfl_xor_sync(0xffffffffu, sl, o);
    dd_add(sh, sl, oh, ol);
    if (WFMT == 0) {
      const float qh = __shfl_xor_sync(0xffffffffu, mh, o), ql = __shfl_xor_sync(0xffffffffu, ml, o);
      pair_max(mh, ml, qh, ql);
    }
  }
  if (lane == 0) wred[warp] = make_float4(sh, sl, mh, ml);
  __syncthreads();
  cluster_wait();  // every CTA of the cluster has initialised its barrier
  if (tid < C) {   // the CTA's partials, to CTA tid
    float th = wred[0].x, tl = wred[0].y, qh = wred[0].z, ql = wred[0].w;
#pragma unroll
    for (int w = 1; w < W; ++w) {
      dd_add(th, tl, wred[w].x, wred[w].y);
      pair_max(qh, ql, wred[w].z, wred[w].w);
    }
    if (WFMT == 0)
      st_async_v4(mapa(smem_u32(&ex1[r]), tid), make_float4(th, tl, qh, ql), mapa(smem_u32(&bar1), tid));
    else
      asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
                       mapa(smem_u32(&ex1[r]), tid)),
                   "f"(th), "f"(tl), "r"(mapa(smem_u32(&bar1), tid))
                   : "memory");
  }
  const bool ok1 = mbar_wait_cluster(&bar1, 0, p.status, wait_limit(p));
  // the C partials combined by a fixed shuffle tree (lane l starts from
  // partial l % C) and taken from lane 0: the same sum and maximum in every
  // warp of every CTA of the cluster
  float th = ex1[lane & (C - 1)].x, tl = ex1[lane & (C - 1)].y;
  float qh = ex1[lane & (C - 1)].z, ql = ex1[lane & (C - 1)].w;
#pragma unroll
  for (int o = C / 2; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, th, o), ol = __shfl_xor_sync(0xffffffffu, tl, o);
    dd_add(th, tl, oh, ol);
    if (WFMT == 0) {
      const float a = __shfl_xor_sync(0xffffffffu, qh, o), b = __shfl_xor_sync(0xffffffffu, ql, o);
      pair_max(qh, ql, a, b);
    }
  }
  th = __shfl_sync(0xffffffffu, th, 0);
  tl = __shfl_sync(0xffffffffu, tl, 0);
  qh = __shfl_sync(0xffffffffu, qh, 0);
  ql = __shfl_sync(0xffffffffu, ql, 0);
  float rh, rl;
  rstd_from_dd(th, tl, H, p.eps, rh, rl);
  if (act && ok1) norm8(acc, gw, rh, rl);
  uint2 *xq = reinterpret_cast<uint2 *>(p.xq + (int64_t)m * H);
  if (WFMT == 0) {
    const float tmax = amax_from_pair(qh, ql, rh, rl);
    const float s = tmax == 0.f ? 1.0f : __fdiv_rn(tmax, kFp8Max);
    if (act && ok1) {  // n * RN(1 / s) where every value within kSafe gives the same code, else n / s
      uint2 w;
      if (!codes8_checked(acc, __frcp_rn(s), w) || p.exact_norm) w = quant8_ptpc(acc, s);
      xq[c] = w;
    }
    if (r == 0 && tid == 0) p.x_scale[m] = s;
  } else {
    float bm = act ? amax8(acc) : 0.f;
    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
    if (act && ok1) {
      const int e = mx_exponent(bm);
      xq[c] = quant8_mx(acc, pow2_neg(e));
      if ((c & 3) == 0) p.xsf[sf128x4_offset(m, c >> 2, ksf)] = (uint8_t)(e + 127);
    }
  }
  if (cs_thread && cpos >= 0 && cpos < p.max_pos) prefetch_l2(p.cos_sin + cpos * kRotDim);
}

__global__ void pa_pack_scales_kernel(const uint8_t *src, uint8_t *dst, int rows, int ksf) {
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
using ProKernel = void (*)(Params, int);
// H <= 16384: 1024 threads need at most 2 chunks, 256 threads at most 8
ProKernel kernel_1024(const Params &p) {
  if (p.weight_fmt == 1) return pa_prologue_kernel<1, 1024, 2>;  // (one chunk spills)
  return p.H <= 8 * 1024 ? pa_prologue_kernel<0, 1024, 1> : pa_prologue_kernel<0, 1024, 2>;
}
ProKernel kernel_256(const Params &p) {
  const int maxc = (p.H + 8 * 256 - 1) / (8 * 256);
  const bool mx = p.weight_fmt == 1;
  if (maxc <= 2) return mx ? pa_prologue_kernel<1, 256, 2> : pa_prologue_kernel<0, 256, 2>;
  if (maxc <= 3) return mx ? pa_prologue_kernel<1, 256, 3> : pa_prologue_kernel<0, 256, 3>;
  if (maxc <= 4) return mx ? pa_prologue_kernel<1, 256, 4> : pa_prologue_kernel<0, 256, 4>;
  return mx ? pa_prologue_kernel<1, 256, 8> : pa_prologue_kernel<0, 256, 8>;
}
}  // namespace

// CTAs an SM holds of the kernel launch_prologue picks for these sizes.
cudaError_t prologue_ctas_per_sm(int H, int weight_fmt, bool wide, int *per_sm) {
  Params p{};
  p.H = H;
  p.weight_fmt = weight_fmt;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, wide ? kernel_1024(p) : kernel_256(p), wide ? 1024 : 256,
                                                       0);
}

cudaError_t launch_prologue(const Params &p, int grid, bool pdl, int early_max, cudaStream_t stream) {
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
  const bool wide = grid <= 64;
  cfg.blockDim = dim3(wide ? 1024 : 256);
  const int mode = !pdl ? 0 : grid <= early_max ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, wide ? kernel_1024(p) : kernel_256(p), p, mode);
}

namespace {
template <int WFMT, int C>
cudaError_t launch_rows(const Params &p, bool pdl, cudaStream_t stream) {
  const int kc = ((p.H + C - 1) / C + 31) / 32 * 32;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(p.M * C);
  // a chunk of 8 elements a thread: 128 * 16 / C threads cover H = 16384;
  // K ranges of up to half that take half the threads (no idle warps at the
  // barriers)
  const bool small = kc <= 8 * 128 * 8 / C;
  cfg.blockDim = dim3(small ? 128 * 8 / C : 128 * 16 / C);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  if (small) return cudaLaunchKernelEx(&cfg, pa_prologue_rows_kernel<WFMT, C, 128 * 8 / C>, p, kc, (int)pdl);
  return cudaLaunchKernelEx(&cfg, pa_prologue_rows_kernel<WFMT, C>, p, kc, (int)pdl);
}

}  // namespace

// Clusters of 8 CTAs a row: measured faster than 16 (6.48 against 6.59 us a
// decode step) and than 4 (6.6-6.8 us): fewer CTAs to launch and complete,
// a shorter exchange, while the arithmetic still spreads over 8 SMs a row.
cudaError_t launch_prologue_rows(const Params &p, bool pdl, cudaStream_t stream) {
  return p.weight_fmt == 0 ? launch_rows<0, 8>(p, pdl, stream) : launch_rows<1, 8>(p, pdl, stream);
}

cudaError_t launch_pack_scales(const uint8_t *src, uint8_t *dst, int rows, int ksf, cudaStream_t stream) {
  const int64_t total = ((int64_t)rows + 127) / 128 * 128 * ksf;
  const int grid = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, pa_pack_scales_kernel, src, dst, rows, ksf);
}

}  // namespace pa
