// Skinny-M path of the pre-attention projection (M <= 16 token rows, the
// decode shapes): an HBM-bound FP8 GEMV over the fused [q|k|v|index_q|index_k]
// weight with the per-head epilogue fused behind it.
//
// Work split: CTA c of G owns output channels [c*N/G, (c+1)*N/G) (balanced to
// one row) over all of K.  A producer warp streams the CTA's weight rows
// through a shared-memory ring with 1-D bulk copies (cp.async.bulk, 512 K
// bytes a row a stage, every stage in flight at once), issued before the
// kernel waits on the prologue (programmatic dependent launch), so the weight
// stream overlaps the prologue and the previous kernel's tail.  Eight consumer
// warps split each 512-byte stage into 64-byte K slices: two e4m3
// m16n8k32 warp MMAs per slice, B columns = tokens (the pre_attn page's GEMV
// tasks put the token on the MFMA B column the same way).  The dot products
// are a few hundred MMAs per CTA, far below the weight stream's time, so the
// legacy MMA is ample here; the dense prefill contraction uses tcgen05.
//
// Per 32-element K block the MXFP8 format rescales each MMA result by
// 2^(e_w + e_x) before accumulating ([EPI] MXFP8 projection); the
// per-channel format scales once at the end by x_scale * w_scale
// ("vllm.models.minimax_m3.amd.mono.kernels.pre_attn", GEMV tasks).
//
// The projection rows go to an f32 scratch in the workspace; the CTA whose
// arrival completes a head's 128 channels (an atomic counter per head, no
// waiting) runs that head's epilogue for every token: one warp per token,
// 4 dims per lane, as the pre_attn page's head tasks.
#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

constexpr int kGvConsumers = 8;
constexpr int kGvThreads = (kGvConsumers + 1) * 32;
constexpr int kChunk = 512;          // K bytes of a ring stage
constexpr int kPitch = kChunk + 32;  // rows 32 B apart modulo 128: conflict-free 8-byte reads
constexpr int kMaxMT = 5;            // up to 80 weight rows per CTA
constexpr int kMaxRows = 16 * kMaxMT;
constexpr int kRingBudget = 108 * 1024;  // two CTAs fit on an SM (overlap of consecutive steps)

template <int WFMT, int NT>
__global__ void __launch_bounds__(kGvThreads) gemv_kernel(Params p, int G, int rmax, int S, int use_pdl) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int fin[8];
  __shared__ int nfin;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N, K = p.H, M = p.M;
  const int r0 = (int)((int64_t)blockIdx.x * N / G), r1 = (int)((int64_t)(blockIdx.x + 1) * N / G);
  const int R = r1 - r0;
  const int MT = (R + 15) >> 4;
  const int nchunks = (K + kChunk - 1) / kChunk;
  const int ksf = K >> 5;
  const int stage_bytes = rmax * kPitch;
  const int ring_bytes = S * stage_bytes;
  const int red_bytes = kGvConsumers * rmax * 16 * 4;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + (ring_bytes > red_bytes ? ring_bytes : red_bytes));
  uint64_t *empty = full + S;
  float *red = reinterpret_cast<float *>(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGvConsumers);
    }
    nfin = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (use_pdl) pdl_trigger();

  float acc[kMaxMT][NT][4];
#pragma unroll
  for (int mt = 0; mt < kMaxMT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;

  if (warp == kGvConsumers) {
    // --------------------------------------------------------- producer warp
    for (int ch = 0; ch < nchunks; ++ch) {
      const int s = ch % S;
      if (ch >= S && !mbar_wait(&empty[s], ((ch / S) - 1) & 1, p.status)) break;
      const int kb0 = ch * kChunk;
      const int bytes = K - kb0 < kChunk ? K - kb0 : kChunk;
      if (lane == 0) mbar_expect_tx(&full[s], (uint32_t)(bytes * R));
      __syncwarp();
      uint8_t *dst = smem + s * stage_bytes;
      for (int r = lane; r < R; r += 32)
        bulk_g2s(dst + r * kPitch, p.w + (int64_t)(r0 + r) * K + kb0, (uint32_t)bytes, &full[s]);
    }
  } else {
    // -------------------------------------------------------- consumer warps
    if (use_pdl) pdl_wait();
    const int g = lane >> 2, t = lane & 3;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int s = ch % S;
      const int kw = ch * kChunk + warp * 64;  // this warp's 64-byte K slice (two 32-blocks)
      const bool active = kw < K;
      // B fragments: token nt*8+g, block b of the slice: bytes kw + 32b + 8t .. + 8
      uint2 bf[NT][2];
      float xs[NT][2][2];  // MXFP8: 2^e_x of tokens nt*8+2t(+1), block b
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tok = nt * 8 + g;
#pragma unroll
        for (int b = 0; b < 2; ++b)
          bf[nt][b] = (active && tok < M)
                          ? __ldcg(reinterpret_cast<const uint2 *>(p.xq + (int64_t)tok * K + kw + 32 * b + 8 * t))
                          : make_uint2(0u, 0u);
        if (WFMT == 1) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            int tk = nt * 8 + 2 * t + j;
            tk = tk < M ? tk : M - 1;
            const uint32_t w2 =
                active ? __ldcg(reinterpret_cast<const unsigned short *>(p.xsf + sf128x4_offset(tk, kw >> 5, ksf)))
                       : 0u;
            xs[nt][0][j] = e8m0_to_f32(w2 & 0xff);
            xs[nt][1][j] = e8m0_to_f32(w2 >> 8);
          }
        }
      }
      if (!mbar_wait(&full[s], (ch / S) & 1, p.status)) break;
      if (active) {
        const uint8_t *st = smem + s * stage_bytes + warp * 64 + 8 * t;
#pragma unroll
        for (int mt = 0; mt < kMaxMT; ++mt) {
          if (mt < MT) {
            const int ra = mt * 16 + g, rb = ra + 8;
            uint2 alo[2], ahi[2];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              alo[b] = ra < R ? *reinterpret_cast<const uint2 *>(st + ra * kPitch + 32 * b) : make_uint2(0u, 0u);
              ahi[b] = rb < R ? *reinterpret_cast<const uint2 *>(st + rb * kPitch + 32 * b) : make_uint2(0u, 0u);
            }
            float ws[2][2];  // MXFP8: 2^e_w of rows ra, rb for block b
            if (WFMT == 1) {
              const int ga = min(r0 + ra, N - 1), gb = min(r0 + rb, N - 1);
              const uint32_t wa = __ldg(reinterpret_cast<const unsigned short *>(p.wsf + sf128x4_offset(ga, kw >> 5, ksf)));
              const uint32_t wb = __ldg(reinterpret_cast<const unsigned short *>(p.wsf + sf128x4_offset(gb, kw >> 5, ksf)));
              ws[0][0] = e8m0_to_f32(wa & 0xff);
              ws[1][0] = e8m0_to_f32(wa >> 8);
              ws[0][1] = e8m0_to_f32(wb & 0xff);
              ws[1][1] = e8m0_to_f32(wb >> 8);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int b = 0; b < 2; ++b) {
                if (WFMT == 0) {
                  mma_e4m3_16832(acc[mt][nt], alo[b].x, ahi[b].x, alo[b].y, ahi[b].y, bf[nt][b].x, bf[nt][b].y);
                } else {
                  float c[4] = {0.f, 0.f, 0.f, 0.f};
                  mma_e4m3_16832(c, alo[b].x, ahi[b].x, alo[b].y, ahi[b].y, bf[nt][b].x, bf[nt][b].y);
                  acc[mt][nt][0] = fmaf(c[0], ws[b][0] * xs[nt][b][0], acc[mt][nt][0]);
                  acc[mt][nt][1] = fmaf(c[1], ws[b][0] * xs[nt][b][1], acc[mt][nt][1]);
                  acc[mt][nt][2] = fmaf(c[2], ws[b][1] * xs[nt][b][0], acc[mt][nt][2]);
                  acc[mt][nt][3] = fmaf(c[3], ws[b][1] * xs[nt][b][1], acc[mt][nt][3]);
                }
              }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  __syncthreads();  // every stage consumed: the ring is free for the reduction

  // --------------------------------------------- cross-warp reduction -> y
  if (warp < kGvConsumers) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mt = 0; mt < kMaxMT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = mt * 16 + g + 8 * (e >> 1), tok = nt * 8 + 2 * t + (e & 1);
          if (mt < MT && row < R) red[(warp * rmax + row) * 16 + tok] = acc[mt][nt][e];
        }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < R * M; i += kGvThreads) {
    const int tok = i / R, row = i - tok * R;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kGvConsumers; ++w) v += red[(w * rmax + row) * 16 + tok];
    if (WFMT == 0) v = v * __ldcg(p.x_scale + tok) * __ldg(p.w_scale + r0 + row);
    __stcg(p.y + (int64_t)tok * N + r0 + row, v);
  }

  // ------------------------------------- arrival; the last CTA of a head runs it
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    for (int h = r0 >> 7; h <= (r1 - 1) >> 7; ++h) {
      const int lo = r0 > (h << 7) ? r0 : (h << 7);
      const int hi = r1 < ((h + 1) << 7) ? r1 : ((h + 1) << 7);
      const int cnt = hi - lo;
      const int old = atomicAdd(p.head_cnt + h, cnt);
      if (old + cnt == kHeadDim) {
        fin[nfin++] = h;
        p.head_cnt[h] = 0;  // every arrival of this launch is in: reset for the next
      }
    }
    __threadfence();
  }
  __syncthreads();
  const int nf = nfin;
  for (int f = 0; f < nf; ++f) {
    const int h = fin[f];
    for (int m = warp; m < M; m += kGvConsumers + 1) {
      HeadCtx hc;
      hc.m = m;
      hc.head = h;
      hc.pos = load_pos(p, m);
      hc.slot = ld_i64(p.slot + m);
      hc.islot = ld_i64(p.islot + m);
      const float4 y4 = __ldcg(reinterpret_cast<const float4 *>(p.y + (int64_t)m * N + h * kHeadDim + 4 * lane));
      float v[4] = {y4.x, y4.y, y4.z, y4.w};
      head_epilogue<4>(p, hc, v, 4 * lane);
    }
  }
}

struct GemvPlan {
  int G, rmax, S, smem;
};

static GemvPlan plan_gemv(const Params &p, int num_sms) {
  GemvPlan g;
  int G = num_sms;
  const int need = (p.N + kMaxRows - 1) / kMaxRows;
  if (G < need) G = need;
  if (G > p.N) G = p.N;
  g.G = G;
  g.rmax = (p.N + G - 1) / G;
  const int stage = g.rmax * kPitch;
  const int nchunks = (p.H + kChunk - 1) / kChunk;
  int S = kRingBudget / stage;
  if (S < 2) S = 2;
  if (S > nchunks) S = nchunks;
  g.S = S;
  const int ring = S * stage, red = kGvConsumers * g.rmax * 16 * 4;
  g.smem = (ring > red ? ring : red) + 2 * S * 8;
  return g;
}

template <int WFMT, int NT>
static cudaError_t launch_gemv_t(const Params &p, const GemvPlan &g, bool pdl, cudaStream_t stream) {
  auto kern = gemv_kernel<WFMT, NT>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), g.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(g.G);
  cfg.blockDim = dim3(kGvThreads);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p, g.G, g.rmax, g.S, (int)pdl);
}

cudaError_t launch_gemv(const Params &p, int num_sms, bool pdl, cudaStream_t stream) {
  const GemvPlan g = plan_gemv(p, num_sms);
  if (p.M <= 8) return p.weight_fmt == 0 ? launch_gemv_t<0, 1>(p, g, pdl, stream) : launch_gemv_t<1, 1>(p, g, pdl, stream);
  return p.weight_fmt == 0 ? launch_gemv_t<0, 2>(p, g, pdl, stream) : launch_gemv_t<1, 2>(p, g, pdl, stream);
}

}  // namespace pa
