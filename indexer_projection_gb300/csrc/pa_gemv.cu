// Skinny-M path of the pre-attention projection (M <= 16 token rows, the
// decode shapes): an HBM-bound FP8 GEMV over the fused [q|k|v|index_q|index_k]
// weight with the per-head epilogue fused behind it.
//
// Work split: CTA c of G owns output channels [c*N/G, (c+1)*N/G) (balanced to
// one row) over all of K.  A producer warp streams the CTA's weight rows
// through a shared-memory ring with 1-D bulk copies (cp.async.bulk, one copy
// a row a stage, 512-1536 K bytes), issued before the kernel waits on the
// prologue (programmatic dependent launch), so the weight stream overlaps the
// prologue and the previous kernel's tail; at the decode shape the whole
// weight slice is in flight at once.  Eight consumer warps own contiguous K
// ranges of each stage; their activation fragments are loaded into registers
// once, right after the wait, so the K loop never waits on L2.  The inner
// products are e4m3 m16n8k32 warp MMAs with the tokens on the B columns (the
// pre_attn page's GEMV tasks put the token on the MFMA B column the same
// way): a few hundred per CTA, far below the weight stream's time, so the
// legacy MMA is ample here; the dense prefill contraction uses tcgen05.
//
// Per 32-element K block the MXFP8 format rescales each MMA result by
// 2^(e_w + e_x) before accumulating ([EPI] MXFP8 projection), with both
// operands' block scales staged in shared memory; the per-channel format
// scales once at the end by x_scale * w_scale
// ("vllm.models.minimax_m3.amd.mono.kernels.pre_attn", GEMV tasks).
//
// The projection rows go to an f32 scratch in the workspace; the CTA whose
// arrival completes a head's 128 channels (an atomic counter per head, no
// waiting) runs that head's epilogue for every token: one warp per token,
// 4 dims per lane, as the pre_attn page's head tasks.  The tokens' positions,
// slots and cos/sin rows and the head gammas are staged in shared memory
// while the weights stream, so the finishing CTA waits only on its rows.
#include "pa_device.cuh"
#include "pa_launch.h"
#include "pa_norm.cuh"

namespace pa {

constexpr int kGvConsumers = 8;
constexpr int kGvThreads = (kGvConsumers + 1) * 32;
constexpr int kSlice = 64;               // K bytes of one MMA pair (two 32-element blocks)
constexpr int kMaxMT = 5;                // up to 80 weight rows per CTA
constexpr int kMaxRows = 16 * kMaxMT;
constexpr int kRingBudget = 108 * 1024;  // two CTAs fit on an SM (overlap of consecutive steps)
constexpr int kBRegSlices = 12;          // activation slices a warp keeps in registers (K <= 6144)
constexpr int kMaxTok = 16;

constexpr int kFusedMaxChunks = 4;       // fused row normalisation: H <= 8 * 288 * 4 = 9216
constexpr int kFusedMaxH = 8 * kGvThreads * kFusedMaxChunks;

struct GvStatic {
  int64_t slot[kMaxTok], islot[kMaxTok];
  __nv_bfloat16 cs[kMaxTok][kRotDim];
  __nv_bfloat16 gam[4][kHeadDim];
  float red[kGvThreads / 32];
  float2 red2[kGvThreads / 32];
  int fin[8];
  int nfin;
};

// FUSED: the step in one launch.  CTAs 0 .. M-1 first normalise and quantise
// token row blockIdx.x (the prologue, pa_norm.cuh) and publish it with a
// release flag; every CTA has its weight stream in flight before that and
// waits (bounded) on the flags of all M rows before its MMAs.  The last CTA
// to finish clears the flags for the next launch.
template <int WFMT, int NT, bool BREG, bool FUSED>
__global__ void __launch_bounds__(kGvThreads, NT == 1 ? 2 : 1)
    gemv_kernel(Params p, int G, int rmax, int S, int chunk, int use_pdl) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ GvStatic sm;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N, K = p.H, M = p.M;
  const int r0 = (int)((int64_t)blockIdx.x * N / G), r1 = (int)((int64_t)(blockIdx.x + 1) * N / G);
  const int R = r1 - r0;
  const int MT = (R + 15) >> 4;
  const int nchunks = (K + chunk - 1) / chunk;
  const int jw = chunk / (kSlice * kGvConsumers);  // slices per warp per chunk
  const int pitch = chunk + 32;                    // rows 32 B apart modulo 128: conflict-free 8-byte reads
  const int ksf = K >> 5;
  const int stage_bytes = rmax * pitch;
  const int ring_bytes = S * stage_bytes;
  const int red_bytes = kGvConsumers * rmax * kMaxTok * 4;
  const int ring_or_red = ring_bytes > red_bytes ? ring_bytes : red_bytes;
  uint8_t *xsf_s = smem + ring_or_red;                  // MXFP8: [M][ksf] token scales
  uint8_t *wsf_s = xsf_s + (WFMT == 1 ? kMaxTok * ksf : 0);  // MXFP8: [R][ksf] weight scales
  uint64_t *full = reinterpret_cast<uint64_t *>(wsf_s + (WFMT == 1 ? ((rmax * ksf + 15) & ~15) : 0));
  uint64_t *empty = full + S;
  float *red = reinterpret_cast<float *>(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGvConsumers);
    }
    sm.nfin = 0;
    fence_mbar_init();
  }
  // static per-layer data may be read before the wait on the previous kernel
  for (int i = threadIdx.x; i < 4 * kHeadDim / 8; i += kGvThreads) {
    const int r = i / (kHeadDim / 8), c = i % (kHeadDim / 8);
    const __nv_bfloat16 *g = r == 0 ? p.g_q : r == 1 ? p.g_k : r == 2 ? p.g_iq : p.g_ik;
    reinterpret_cast<uint4 *>(sm.gam[r])[c] = __ldg(reinterpret_cast<const uint4 *>(g) + c);
  }
  if (WFMT == 1) {  // this CTA's weight-row block scales, F8_128x4 -> [row][kb]
    for (int i = threadIdx.x; i < R * (ksf >> 2); i += kGvThreads) {
      const int row = i / (ksf >> 2), kq = i - row * (ksf >> 2);
      *reinterpret_cast<uint32_t *>(wsf_s + row * ksf + 4 * kq) =
          __ldg(reinterpret_cast<const uint32_t *>(p.wsf + sf128x4_offset(r0 + row, 4 * kq, ksf)));
    }
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

  // weights (static) stream before the wait on the previous kernel
  auto issue = [&](const int ch) {
    const int s = ch % S;
    const int kb0 = ch * chunk;
    const int bytes = K - kb0 < chunk ? K - kb0 : chunk;
    if (lane == 0) mbar_expect_tx(&full[s], (uint32_t)(bytes * R));
    __syncwarp();
    uint8_t *dst = smem + s * stage_bytes;
    for (int r = lane; r < R; r += 32)
      bulk_g2s(dst + r * pitch, p.w + (int64_t)(r0 + r) * K + kb0, (uint32_t)bytes, &full[s]);
  };
  const int first = S < nchunks ? S : nchunks;
  if (warp == kGvConsumers)
    for (int ch = 0; ch < first; ++ch) issue(ch);
  if (use_pdl) pdl_wait();
  if (FUSED) {
    if (blockIdx.x < M) {  // this CTA normalises token row blockIdx.x
      norm_quant_row<WFMT, kGvThreads, kFusedMaxChunks>(p, blockIdx.x, sm.red, sm.red2);
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();
        st_release(p.row_flag + blockIdx.x, 1);
      }
    }
  }
  // per-step data the epilogue needs, staged while the weights stream
  if (warp == 0 && lane < M) {
    const int64_t pos = load_pos(p, lane);
    sm.slot[lane] = ld_i64(p.slot + lane);
    sm.islot[lane] = ld_i64(p.islot + lane);
    const uint4 *src = reinterpret_cast<const uint4 *>(p.cos_sin + pos * kRotDim);
#pragma unroll
    for (int c = 0; c < kRotDim / 8; ++c) reinterpret_cast<uint4 *>(sm.cs[lane])[c] = __ldg(src + c);
  }
  if (FUSED) {  // every row's activations published
    if (threadIdx.x < M) {
      const int *f = p.row_flag + threadIdx.x;
      if (ld_acquire(f) != 1) {
        const uint64_t t0 = globaltimer();
        while (ld_acquire(f) != 1) {
          if (globaltimer() - t0 > 1000000000ull) {
            set_status(p.status, kDevWaitTimeout);
            break;
          }
          __nanosleep(64);
        }
      }
    }
    __syncthreads();
  }
  if (WFMT == 1) {  // the tokens' block scales, F8_128x4 -> [tok][kb]
    for (int i = threadIdx.x; i < M * (ksf >> 2); i += kGvThreads) {
      const int tok = i / (ksf >> 2), kq = i - tok * (ksf >> 2);
      *reinterpret_cast<uint32_t *>(xsf_s + tok * ksf + 4 * kq) =
          __ldcg(reinterpret_cast<const uint32_t *>(p.xsf + sf128x4_offset(tok, 4 * kq, ksf)));
    }
    __syncthreads();
  }

  if (warp == kGvConsumers) {
    // ------------------------------------------------ producer warp: refills
    for (int ch = first; ch < nchunks; ++ch) {
      if (!mbar_wait(&empty[ch % S], ((ch / S) - 1) & 1, p.status)) break;
      issue(ch);
    }
  } else {
    // -------------------------------------------------------- consumer warps
    const int g = lane >> 2, t = lane & 3;
    // activation fragments of every slice of this warp: token nt*8+g, block b
    // of the slice: bytes kw + 32b + 8t .. + 8
    uint2 bpre[BREG ? kBRegSlices : 1][NT][2];
    if (BREG) {
#pragma unroll
      for (int sl = 0; sl < kBRegSlices; ++sl) {
        const int ch = sl / jw, i = sl - ch * jw;
        const int kw = ch * chunk + warp * (chunk / kGvConsumers) + kSlice * i;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int tok = nt * 8 + g;
#pragma unroll
          for (int b = 0; b < 2; ++b)
            bpre[sl][nt][b] = (sl < nchunks * jw && kw < K && tok < M)
                                  ? __ldcg(reinterpret_cast<const uint2 *>(p.xq + (int64_t)tok * K + kw + 32 * b + 8 * t))
                                  : make_uint2(0u, 0u);
        }
      }
    }
    // one pass over this warp's slices; slice sl sits in chunk sl / jw
    const int nsl = nchunks * jw;
    bool alive = true;
    auto slice = [&](const int sl, const uint2 (&bf)[NT][2]) {
      const int ch = sl / jw, i = sl - ch * jw, s = ch % S;
      if (i == 0 && alive) alive = mbar_wait(&full[s], (ch / S) & 1, p.status);
      const int kw = ch * chunk + warp * (chunk / kGvConsumers) + kSlice * i;
      if (alive && kw < K) {
        float xs[NT][2][2];  // MXFP8: 2^e_x of tokens nt*8+2t(+1), block b
        if (WFMT == 1) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              int tk = nt * 8 + 2 * t + j;
              tk = tk < M ? tk : M - 1;
              const uint32_t w2 = *reinterpret_cast<const unsigned short *>(xsf_s + tk * ksf + (kw >> 5));
              xs[nt][0][j] = e8m0_to_f32(w2 & 0xff);
              xs[nt][1][j] = e8m0_to_f32(w2 >> 8);
            }
        }
        const uint8_t *st = smem + s * stage_bytes + (kw - ch * chunk) + 8 * t;
#pragma unroll
        for (int mt = 0; mt < kMaxMT; ++mt) {
          if (mt < MT) {
            const int ra = mt * 16 + g, rb = ra + 8;
            uint2 alo[2], ahi[2];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              alo[b] = ra < R ? *reinterpret_cast<const uint2 *>(st + ra * pitch + 32 * b) : make_uint2(0u, 0u);
              ahi[b] = rb < R ? *reinterpret_cast<const uint2 *>(st + rb * pitch + 32 * b) : make_uint2(0u, 0u);
            }
            float ws[2][2];  // MXFP8: 2^e_w of rows ra, rb for block b
            if (WFMT == 1) {
              const int ca = ra < R ? ra : R - 1, cb = rb < R ? rb : R - 1;
              const uint32_t wa = *reinterpret_cast<const unsigned short *>(wsf_s + ca * ksf + (kw >> 5));
              const uint32_t wb = *reinterpret_cast<const unsigned short *>(wsf_s + cb * ksf + (kw >> 5));
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
      if (i == jw - 1 || sl == nsl - 1) {  // the warp is done with this stage
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    };
    if (BREG) {
#pragma unroll
      for (int sl = 0; sl < kBRegSlices; ++sl)
        if (sl < nsl) slice(sl, bpre[sl]);
    } else {
      for (int sl = 0; sl < nsl; ++sl) {
        const int ch = sl / jw, i = sl - ch * jw;
        const int kw = ch * chunk + warp * (chunk / kGvConsumers) + kSlice * i;
        uint2 bf[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int tok = nt * 8 + g;
#pragma unroll
          for (int b = 0; b < 2; ++b)
            bf[nt][b] = (tok < M && kw < K)
                            ? __ldcg(reinterpret_cast<const uint2 *>(p.xq + (int64_t)tok * K + kw + 32 * b + 8 * t))
                            : make_uint2(0u, 0u);
        }
        slice(sl, bf);
      }
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
          if (mt < MT && row < R) red[(warp * rmax + row) * kMaxTok + tok] = acc[mt][nt][e];
        }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < R * M; i += kGvThreads) {
    const int tok = i / R, row = i - tok * R;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kGvConsumers; ++w) v += red[(w * rmax + row) * kMaxTok + tok];
    if (WFMT == 0) v = v * __ldcg(p.x_scale + tok) * __ldg(p.w_scale + r0 + row);
    __stcg(p.y + (int64_t)tok * N + r0 + row, v);
  }
  __threadfence();  // release this thread's rows before the CTA's arrival is counted

  // ------------------------------------- arrival; the last CTA of a head runs it
  __syncthreads();
  const int h0 = r0 >> 7, nh = ((r1 - 1) >> 7) - h0 + 1;
  if (threadIdx.x < nh) {
    const int h = h0 + threadIdx.x;
    const int lo = r0 > (h << 7) ? r0 : (h << 7);
    const int hi = r1 < ((h + 1) << 7) ? r1 : ((h + 1) << 7);
    const int cnt = hi - lo;
    const int old = atomicAdd(p.head_cnt + h, cnt);
    if (old + cnt == kHeadDim) {
      sm.fin[atomicAdd(&sm.nfin, 1)] = h;
      p.head_cnt[h] = 0;  // every arrival of this launch is in: reset for the next
      __threadfence();    // acquire the other CTAs' rows
    }
  }
  __syncthreads();
  const int nf = sm.nfin;
  for (int f = 0; f < nf; ++f) {
    const int h = sm.fin[f];
    for (int m = warp; m < M; m += kGvConsumers + 1) {
      HeadCtx hc;
      hc.m = m;
      hc.head = h;
      hc.slot = sm.slot[m];
      hc.islot = sm.islot[m];
      hc.cs_row = sm.cs[m];
      hc.g_q = sm.gam[0];
      hc.g_k = sm.gam[1];
      hc.g_iq = sm.gam[2];
      hc.g_ik = sm.gam[3];
      const float4 y4 = __ldcg(reinterpret_cast<const float4 *>(p.y + (int64_t)m * N + h * kHeadDim + 4 * lane));
      float v[4] = {y4.x, y4.y, y4.z, y4.w};
      head_epilogue<4>(p, hc, v, 4 * lane);
    }
  }
  if (FUSED) {  // the last CTA out clears the row flags for the next launch
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(p.done_cnt, 1) == G - 1) {
        for (int m = 0; m < M; ++m) p.row_flag[m] = 0;
        *p.done_cnt = 0;
        __threadfence();
      }
    }
  }
}

struct GemvPlan {
  int G, rmax, S, chunk, smem;
  bool breg;
};

static GemvPlan plan_gemv(const Params &p, int num_sms) {
  GemvPlan g;
  int G = num_sms;
  const int need = (p.N + kMaxRows - 1) / kMaxRows;
  if (G < need) G = need;
  if (G > p.N) G = p.N;
  g.G = G;
  g.rmax = (p.N + G - 1) / G;
  // the largest stage (1536, 1024 or 512 K bytes a row) whose ring holds at
  // least min(4, stages) stages in the budget
  g.chunk = 512;
  g.S = 1;
  for (int j = 3; j >= 1; --j) {
    const int chunk = 512 * j;
    const int nchunks = (p.H + chunk - 1) / chunk;
    int S = kRingBudget / (g.rmax * (chunk + 32));
    if (S > nchunks) S = nchunks;
    if (S >= (nchunks < 4 ? nchunks : 4) || j == 1) {
      g.chunk = chunk;
      g.S = S < 1 ? 1 : S;
      break;
    }
  }
  g.breg = p.H / 512 <= kBRegSlices;
  const int ring = g.S * g.rmax * (g.chunk + 32), red = kGvConsumers * g.rmax * kMaxTok * 4;
  const int ksf = p.H / 32;
  const int scales = p.weight_fmt == 1 ? kMaxTok * ksf + ((g.rmax * ksf + 15) & ~15) : 0;
  g.smem = (ring > red ? ring : red) + scales + 2 * g.S * 8;
  return g;
}

template <int WFMT, int NT, bool BREG, bool FUSED>
static cudaError_t launch_gemv_t(const Params &p, const GemvPlan &g, bool pdl, cudaStream_t stream) {
  auto kern = gemv_kernel<WFMT, NT, BREG, FUSED>;
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
  return cudaLaunchKernelEx(&cfg, kern, p, g.G, g.rmax, g.S, g.chunk, (int)pdl);
}

template <int WFMT, int NT>
static cudaError_t launch_gemv_b(const Params &p, const GemvPlan &g, bool pdl, bool fused, cudaStream_t stream) {
  if (fused)  // fused implies H <= 9216, so the activations fit in registers
    return launch_gemv_t<WFMT, NT, true, true>(p, g, pdl, stream);
  return g.breg ? launch_gemv_t<WFMT, NT, true, false>(p, g, pdl, stream)
                : launch_gemv_t<WFMT, NT, false, false>(p, g, pdl, stream);
}

bool gemv_fuses_prologue(const Params &p) { return p.M <= kMaxTok && p.H <= kFusedMaxH && p.H <= 512 * kBRegSlices; }

cudaError_t launch_gemv(const Params &p, int num_sms, bool pdl, bool fused, cudaStream_t stream) {
  const GemvPlan g = plan_gemv(p, num_sms);
  if (p.M <= 8)
    return p.weight_fmt == 0 ? launch_gemv_b<0, 1>(p, g, pdl, fused, stream) : launch_gemv_b<1, 1>(p, g, pdl, fused, stream);
  return p.weight_fmt == 0 ? launch_gemv_b<0, 2>(p, g, pdl, fused, stream) : launch_gemv_b<1, 2>(p, g, pdl, fused, stream);
}

}  // namespace pa
