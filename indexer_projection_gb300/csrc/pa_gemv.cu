// Skinny-M path of the pre-attention projection (M <= 16 token rows, the
// decode shapes): an HBM-bound FP8 GEMV over the fused [q|k|v|index_q|index_k]
// weight on the tcgen05 tensor cores, one thread-block cluster per 128-channel
// head, with the head's epilogue fused behind it.
//
// Work split.  The C CTAs of head h's cluster (C = 16, or 8 where the device
// cannot co-schedule clusters of 16) each own the head's 128 weight rows over
// one K range of kc = ceil(K / C) bytes rounded up to 128 (384 at K = 6144).
// Every thread copies its share of the range's weight rows from HBM straight
// into shared memory with 16-byte cp.async (no registers held), in the
// 128-byte-swizzled K-major layout the tensor core reads, all issued before
// the kernel waits on the prologue (programmatic dependent launch), so the
// weight stream overlaps the prologue.  After the wait the CTA stages the
// range's activations the same way and one thread issues the MMAs:
// tcgen05.mma m128 n16 k32 per 32 bytes of K, weights as A (128 rows),
// tokens as B (16 columns, the absent ones zero), f32 accumulators in tensor
// memory (one per staged chunk, so the MMA chains overlap) (kind::f8f6f4; for MXFP8 kind::mxf8f6f4.block_scale with the
// F8_128x4 scale atoms of both operands moved to tensor memory by
// tcgen05.cp).  A K range longer than the 3 staged 128-byte chunks is
// streamed in batches.  The pre_attn page's GEMV tasks put the token on the
// MFMA B column the same way.
//
// Per 32-element K block the MXFP8 format scales each product by
// 2^(e_w + e_x) inside the MMA ([EPI] MXFP8 projection); the per-channel
// format scales the summed rows by x_scale * w_scale
// ("vllm.models.minimax_m3.amd.mono.kernels.pre_attn", GEMV tasks).
//
// Reduction and epilogue, inside the cluster: warps 0-3 read the 128 x 16
// accumulator (thread = weight row) and store each token m's partial rows
// into the shared memory of cluster CTA m % C with asynchronous
// distributed-shared-memory stores that count their bytes on that CTA's
// mbarrier (no fences, no arrivals).  CTA m % C, once all C x 512 bytes of
// the token's partials are in, sums the C K-range partials of the head's 128
// channels and runs the head epilogue for token m, one warp, 4 dims a lane,
// as the pre_attn page's head tasks.  Nothing goes through global memory
// between the MMAs and the outputs.
//
// Fused variant (clusters of 16, K <= 16 x 384): the kernel also does the
// prologue's work, so the decode step is one launch.  The 16 threads of
// token group m of every CTA add ar + res over the CTA's K range (the
// residual is written by head 0's cluster), reduce sum(acc^2) as a
// double-float, and for the per-channel format the maximum of |acc (1 +
// gam)| (the row's amax before the factor rstd), and exchange the 16 K-range
// partials across the cluster in one st.async each (byte-counted); every CTA
// then combines them in the same order, so all agree bit for bit on rstd and
// the scale.  The correctly rounded n (pa_norm.cuh) gives the FP8 codes,
// written straight into the MMA's B operand (and the MXFP8 scale atoms into
// their tcgen05.cp source): nothing goes through global memory between the
// inputs and the outputs.  The rows' inputs are prefetched into L2 before
// the wait (a hint: the loads after it still see the producer's writes).
//
// The weight, its scales, the head's gamma and w_scale are read before the
// wait on the previous kernel: they must not be written by work still in
// flight on the stream (they are model constants).  Everything else is read
// after the wait.  Every mbarrier wait is bounded (about a second; then
// PA_DEV_WAIT_TIMEOUT), and the tensor memory is freed on every path.
#include "pa_device.cuh"
#include "pa_launch.h"
#include "pa_norm.cuh"
#include "pa_tc.cuh"

namespace pa {

constexpr int kGvThreads = 256;
constexpr int kChunk = 128;        // K bytes of one swizzle atom column (4 MMAs)
constexpr int kStageChunks = 3;    // weight chunks staged at once (48 KB)
constexpr int kWChunkBytes = kHeadDim * kChunk;  // 16 KB: 128 rows x 128 B
constexpr int kXChunkBytes = 16 * kChunk;        // 2 KB: 16 token rows x 128 B
constexpr int kSfAtom = 512;       // F8_128x4: 128 rows x 4 K-blocks
constexpr int kMaxTok = 16;
// Tensor memory (128 columns).  Weights read from shared memory: one
// 16-column accumulator per staged chunk (independent MMA chains, summed when
// read back), scale factors after them.  Per-channel weights of a K range
// that fits one batch are first copied into tensor memory (before the wait
// on the prologue), so the MMAs after it read only the activations from
// shared memory: two accumulators, then the 12 x 8 columns of A.
constexpr int kTmemCols = 128;
constexpr int kSfaCol = 16 * kStageChunks, kSfbCol = kSfaCol + 4;
constexpr int kTaCol = 32;           // A in tensor memory: column kTaCol + 8q for MMA q
constexpr uint32_t kIdescF8 = idesc_f8(128, 16);
constexpr uint32_t kIdescMx = idesc_mx(128, 16);
constexpr int kFusedMaxKc = 384;   // fused variant: 3 chunks of 8 elements a thread

// Byte offsets of the dynamic shared memory from its 1024-aligned base.
struct GvLayout {
  int w;     // [kStageChunks] weight chunks, 128 rows x 128 B, 128B-swizzled
  int x;     // [nchunks] activation chunks, 16 rows x 128 B, 128B-swizzled
  int sfa;   // MXFP8 [kStageChunks] weight scale atoms
  int sfb;   // MXFP8 [nchunks] activation scale atoms
  int recv;  // [TS][C][128] f32 partial rows received from the cluster
  int ex1;   // fused: [16 K ranges][16 tokens] float4 partials: sum(acc^2), max |acc (1 + gam)|
  int gin;   // fused: the K range's input-norm gamma (bf16)
  int total;
};
__host__ __device__ inline GvLayout gv_layout(int C, int kc, int mx) {
  GvLayout L;
  const int nch = kc / kChunk;
  const int ts = (kMaxTok + C - 1) / C;
  L.w = 0;
  L.x = L.w + kStageChunks * kWChunkBytes;
  L.sfa = L.x + nch * kXChunkBytes;
  L.sfb = L.sfa + (mx ? kStageChunks * kSfAtom : 0);
  L.recv = L.sfb + (mx ? nch * kSfAtom : 0);
  L.ex1 = L.recv + ts * C * kHeadDim * 4;
  L.gin = L.ex1 + 16 * kMaxTok * 16;
  L.total = L.gin + kc * 2;
  return L;
}

// Small per-CTA state (static shared memory).
struct alignas(16) GvStatic {  // cs rows are 16-byte cp.async destinations
  float wsc[kHeadDim];           // per-channel weight scales of the head
  __nv_bfloat16 gam[kHeadDim];   // the head role's gamma
  __nv_bfloat16 cs[2][kRotDim];  // cos / sin rows of the tokens finished here
  float xs[kMaxTok];             // per-token activation scales
  int64_t slot[2], islot[2];
  uint64_t mma_bar;              // the MMAs of a batch have completed
  uint64_t recv_bar;             // partial rows received (transaction bytes)
  uint64_t ex1_bar;              // fused: the cluster's norm partials received
  uint64_t never_bar;            // testing (PA_FLAG_TEST_WAIT_TIMEOUT): nothing arrives on it
  uint32_t tmem;
  int ok;
};

// 128B swizzle: 16-byte chunk c of row r of an 8-row, 1024-byte atom.
__device__ __forceinline__ int swz(int r, int c) { return (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ void st_async_b32(uint32_t caddr, float v, uint32_t cbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(caddr),
               "r"(__float_as_uint(v)), "r"(cbar)
               : "memory");
}

// The fused variant's row normalisation for the CTA's K range [k0, k1) of
// every token (G threads a token, G = 32 for up to 8 tokens, else 16: thread
// (m, sub) holds chunks sub + G j of 8 elements), written as the MMA's B
// operand.  Exchanges with the 16 CTAs of the cluster; leaves the per-token
// scales in xs (per-channel format).  The codes come from the checked fast
// path of the many-row prologue (pa_norm.cuh: a cheap n, kept where every
// value within kSafe of it gives the same code or block exponent, else the
// exact n), so they are the exact path's bit for bit.
template <int WFMT>
__device__ __forceinline__ void fused_norm_quant(const Params &p, int tid, int ks, int k0, int k1, int h,
                                                 uint8_t *x_s, uint8_t *sfb_s, float4 *ex1, const uint4 *gin_s,
                                                 float *xs, uint64_t *ex1_bar) {
  constexpr int kJ = kFusedMaxKc / 8 / 16;  // chunks a thread at most (G = 16)
  const int M = p.M, K = p.H;
  const int G = M <= 8 ? 32 : 16;
  const int m = tid / G, sub = tid % G;
  const int cpt = (k1 - k0) / 8;  // chunks of 8 elements a token in the range
  const bool active = m < M;
  float acc[kJ][8];
  float sh = 0.f, sl = 0.f, mh = 0.f, ml = 0.f;
  if (active) {
    const uint4 *ar = reinterpret_cast<const uint4 *>(p.ar + (int64_t)m * K + k0);
    const uint4 *res = reinterpret_cast<const uint4 *>(p.res + (int64_t)m * K + k0);
    uint4 *rout = (h == 0 && p.residual) ? reinterpret_cast<uint4 *>(p.residual + (int64_t)m * K + k0) : nullptr;
    uint4 av[kJ], rv[kJ];  // every load in flight before the first use
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int c = sub + G * j;
      if (c < cpt) {
        av[j] = __ldcs(ar + c);
        rv[j] = __ldcs(res + c);
      }
    }
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int c = sub + G * j;
      if (c < cpt) {
        uint4 rb;
        acc8(av[j], rv[j], acc[j], rb, sh, sl);
        if (rout) __stcs(rout + c, rb);
        if (WFMT == 0) absprod_max8(acc[j], gin_s[c], mh, ml);
      }
    }
  }
  // the token's partials over this K range, in all G lanes of the group
  for (int o = G / 2; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, sh, o), ol = __shfl_xor_sync(0xffffffffu, sl, o);
    dd_add(sh, sl, oh, ol);
    if (WFMT == 0) {
      const float qh = __shfl_xor_sync(0xffffffffu, mh, o), ql = __shfl_xor_sync(0xffffffffu, ml, o);
      pair_max(mh, ml, qh, ql);
    }
  }
  cluster_wait();  // every CTA of the cluster has initialised its barriers
  // lane sub < 16 of token m's group sends this range's partials to cluster CTA sub
  if (active && sub < 16) {
    float4 *dst = ex1 + ks * kMaxTok + m;
    if (WFMT == 0)
      st_async_v4(mapa(smem_u32(dst), sub), make_float4(sh, sl, mh, ml), mapa(smem_u32(ex1_bar), sub));
    else
      asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
                       mapa(smem_u32(dst), sub)),
                   "f"(sh), "f"(sl), "r"(mapa(smem_u32(ex1_bar), sub))
                   : "memory");
  }
  const bool ok1 = mbar_wait_cluster(ex1_bar, 0, p.status, wait_limit(p));
  float rh = 0.f, rl = 0.f;
  if (active && ok1) {
    float th = ex1[m].x, tl = ex1[m].y;  // the 16 K ranges in order: the same sum in every CTA
#pragma unroll
    for (int q = 1; q < 16; ++q) dd_add(th, tl, ex1[q * kMaxTok + m].x, ex1[q * kMaxTok + m].y);
    rstd_from_dd(th, tl, K, p.eps, rh, rl);
  }
  const float f = __fadd_rn(rh, rl);
  // quantise into the B operand: chunk c of token m is K bytes 8c .. 8c + 7 of
  // the range: 128-byte chunk c / 16, 16-byte piece (c % 16) / 2, half c % 2
  auto put = [&](int c, uint2 w) {
    *reinterpret_cast<uint2 *>(x_s + (c >> 4) * kXChunkBytes + swz(m, (c & 15) >> 1) + 8 * (c & 1)) = w;
  };
  if (WFMT == 0) {
    if (active && ok1) {
      float qh = ex1[m].z, ql = ex1[m].w;
#pragma unroll
      for (int q = 1; q < 16; ++q) pair_max(qh, ql, ex1[q * kMaxTok + m].z, ex1[q * kMaxTok + m].w);
      const float tmax = amax_from_pair(qh, ql, rh, rl);
      const float s = tmax == 0.f ? 1.0f : __fdiv_rn(tmax, kFp8Max);
      const float rs = __frcp_rn(s);
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        const int c = sub + G * j;
        if (c < cpt) {
          float t[8];
          napprox8(acc[j], gin_s[c], f, t);
          uint2 w;
          if (!codes8_checked(t, rs, w)) {  // near a code boundary: the exact n and a true divide
            norm8(acc[j], gin_s[c], rh, rl);
            w = quant8_ptpc(acc[j], s);
          }
          put(c, w);
        }
      }
      if (sub == 0) xs[m] = s;
    }
  } else {
    // a 32-element block is 4 consecutive chunks: lanes sub .. sub + 3 of the group
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int c = sub + G * j;
      const bool mine = active && ok1 && c < cpt;
      float t[8];
      float bm = 0.f;
      if (mine) {
        napprox8(acc[j], gin_s[c], f, t);
        bm = amax8(t);
      }
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      // the exponent is exact where every amax within kSafe gives it
      const bool e_ok = mx_exponent(bm * (1.0f - kSafe)) == mx_exponent(bm * (1.0f + kSafe));
      const bool exact = __any_sync(0xffffffffu, !e_ok);  // warp-uniform
      if (exact) {  // rare: this warp's blocks from the exact n (acc[j] becomes n)
        if (mine) {
          norm8(acc[j], gin_s[c], rh, rl);
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = acc[j][i];
        }
        bm = mine ? amax8(t) : 0.f;
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      }
      if (mine) {
        const int e = mx_exponent(bm);
        uint2 w;
        if (!codes8_checked(t, pow2_neg(e), w)) {  // near a code boundary: from the exact n
          if (!exact) norm8(acc[j], gin_s[c], rh, rl);
          w = quant8_mx(acc[j], pow2_neg(e));
        }
        put(c, w);
        // F8_128x4 atom of 128-byte chunk c / 16: row m, K-block (c / 4) % 4
        if ((c & 3) == 0) sfb_s[(c >> 4) * kSfAtom + m * 16 + ((c >> 2) & 3)] = (uint8_t)(e + 127);
      }
    }
  }
}

template <int WFMT, int C, bool FUSED, int CF>
__global__ void __launch_bounds__(kGvThreads, 3) pa_skinny_proj_kernel(Params p, int kc, int use_pdl) {
  static_assert(!FUSED || C == 16, "the fused variant exchanges norm partials among 16 K ranges");
  constexpr int TS = (kMaxTok + C - 1) / C;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t *dsm = dsm_raw + ((1024 - (smem_u32(dsm_raw) & 1023)) & 1023);
  __shared__ GvStatic ss;
  const GvLayout L = gv_layout(C, kc, WFMT);
  uint8_t *w_s = dsm + L.w, *x_s = dsm + L.x, *sfa_s = dsm + L.sfa, *sfb_s = dsm + L.sfb;
  float *recv = reinterpret_cast<float *>(dsm + L.recv);
  float4 *ex1 = reinterpret_cast<float4 *>(dsm + L.ex1);
  uint4 *gin_s = reinterpret_cast<uint4 *>(dsm + L.gin);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = p.H, M = p.M, ksf = K >> 5;
  const int ks = (int)cta_rank();  // this CTA's K range
  const int h = blockIdx.x / C;
  const int k0 = ks * kc, k1 = k0 + kc < K ? k0 + kc : K;
  const int nch = k1 > k0 ? (k1 - k0) / kChunk : 0;

  if (tid == 0) {
    int ntok = 0;  // tokens rank + C * j < M finished here; 512 bytes from each CTA for each
    for (int j = 0; j < TS; ++j) ntok += ks + C * j < M;
    mbar_init(&ss.mma_bar, 1);
    mbar_init(&ss.recv_bar, 1);
    if (ntok) mbar_expect_tx(&ss.recv_bar, (uint32_t)(ntok * C * kHeadDim * 4));
    else mbar_arrive(&ss.recv_bar);
    if (FUSED) {  // every CTA sends 16 (MXFP8: 8) bytes per token to every CTA
      mbar_init(&ss.ex1_bar, 1);
      mbar_expect_tx(&ss.ex1_bar, (uint32_t)(16 * M * (WFMT == 0 ? 16 : 8)));
    }
    mbar_init(&ss.never_bar, 1);
    ss.ok = 1;
    fence_mbar_init();
  }
  if (warp == 4) tc_alloc(&ss.tmem, kTmemCols);
  cluster_arrive_relaxed();  // matched by cluster_wait() before the first remote store

  // ------------------------------- the weight stream (batch 0), before the wait
  const uint8_t *wrow = p.w + (int64_t)h * kHeadDim * K + k0;  // row 0 of the head, this range
  auto issue_weights = [&](int c0) {
    const int n = nch - c0 < kStageChunks ? nch - c0 : kStageChunks;
    for (int i = tid; i < n * kHeadDim * 8; i += kGvThreads) {
      const int j = i / (kHeadDim * 8), rc = i - j * (kHeadDim * 8), r = rc >> 3, c = rc & 7;
      cp_async16(w_s + j * kWChunkBytes + swz(r, c), wrow + (int64_t)r * K + (c0 + j) * kChunk + 16 * c);
    }
    if (WFMT == 1)
      for (int i = tid; i < n * (kSfAtom / 16); i += kGvThreads) {
        const int j = i / (kSfAtom / 16), c = i - j * (kSfAtom / 16);
        cp_async16(sfa_s + j * kSfAtom + 16 * c,
                   p.wsf + ((int64_t)h * (ksf >> 2) + (k0 / kChunk) + c0 + j) * kSfAtom + 16 * c);
      }
    cp_async_commit();
  };
  if (FUSED && (tid >> 4) < M)  // the rows' inputs over this K range: a hint before the wait,
                                // issued ahead of the weight stream
    for (int c = tid & 15; c < (k1 - k0) / 8; c += 16) {
      prefetch_l2(p.ar + (int64_t)(tid >> 4) * K + k0 + 8 * c);
      prefetch_l2(p.res + (int64_t)(tid >> 4) * K + k0 + 8 * c);
    }
  if (FUSED) {  // the K range's input-norm gamma (a model constant), its own group
    for (int i = tid; i < (k1 - k0) / 8; i += kGvThreads) cp_async16(gin_s + i, p.g_in + k0 + 8 * i);
    cp_async_commit();
  }
  issue_weights(0);
  if (FUSED) {  // token rows >= M of the B operand are zero; their scales 2^0
    for (int i = tid; i < nch * kXChunkBytes / 16; i += kGvThreads)
      reinterpret_cast<uint4 *>(x_s)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (WFMT == 1)
      for (int i = tid; i < nch * kSfAtom / 16; i += kGvThreads)
        reinterpret_cast<uint4 *>(sfb_s)[i] = make_uint4(0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
  }
  const bool is_v = h >= p.v0 && h < p.iq0;
  if (tid < 32) {
    if (WFMT == 0)
      reinterpret_cast<float4 *>(ss.wsc)[tid] = __ldg(reinterpret_cast<const float4 *>(p.w_scale + h * kHeadDim) + tid);
  } else if (tid < 48) {
    if (!is_v) {
      const __nv_bfloat16 *gsrc = h < p.k0 ? p.g_q : h < p.v0 ? p.g_k : h < p.ik0 ? p.g_iq : p.g_ik;
      reinterpret_cast<uint4 *>(ss.gam)[tid - 32] = __ldg(reinterpret_cast<const uint4 *>(gsrc) + (tid - 32));
    }
  }
  if (FUSED) cp_async_wait<1>();  // the gamma (the weights stay in flight)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ss.tmem;
  // per-channel weights of a single batch: into tensor memory while the
  // prologue runs (the copies complete before the MMAs issued after them)
  const bool a_tmem = WFMT == 0 && nch > 0 && nch <= kStageChunks;
  if (a_tmem) {
    cp_async_wait<0>();  // this thread's weight copies
    fence_proxy_async_smem();
    __syncthreads();
    if (warp == 4 && lane == 0) {
      tc_fence_after();
      for (int q = 0; q < 4 * nch; ++q)
        tc_cp_128x256b(tmem + kTaCol + 8 * q, sdesc_sw128(smem_u32(w_s + (q >> 2) * kWChunkBytes)) + 2 * (q & 3));
    }
  }
  if (warp == 7 && lane < TS && ks + C * lane < M) {  // inputs: a hint before the wait
    prefetch_l2(p.pos + ks + C * lane);
    prefetch_l2(p.slot + ks + C * lane);
    prefetch_l2(p.islot + ks + C * lane);
  }
  if (use_pdl) {
    pdl_trigger();
    pdl_wait();
  }
  // ------------------------------------------ activations and per-token data
  if (!FUSED) {
    for (int i = tid; i < nch * 16 * 8; i += kGvThreads) {
      const int j = i >> 7, rc = i & 127, r = rc >> 3, c = rc & 7;
      uint8_t *dst = x_s + j * kXChunkBytes + swz(r, c);
      if (r < M) cp_async16(dst, p.xq + (int64_t)r * K + k0 + j * kChunk + 16 * c);
      else *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (WFMT == 1)
      for (int i = tid; i < nch * (kSfAtom / 16); i += kGvThreads) {
        const int j = i / (kSfAtom / 16), c = i - j * (kSfAtom / 16);
        cp_async16(sfb_s + j * kSfAtom + 16 * c, p.xsf + ((int64_t)(k0 / kChunk) + j) * kSfAtom + 16 * c);
      }
    if (WFMT == 0 && tid < M) cp_async4(&ss.xs[tid], p.x_scale + tid);
  }
  // tokens finished here: ks + C * j, j < TS
  const bool cs_lane = warp == 7 && lane < 8 * TS && ks + C * (lane >> 3) < M;
  int64_t pos = 0;
  if (cs_lane) pos = ld_i64(p.pos + ks + C * (lane >> 3));
  if (warp == 7 && lane < TS && ks + C * lane < M) {
    cp_async8(&ss.slot[lane], p.slot + ks + C * lane);
    cp_async8(&ss.islot[lane], p.islot + ks + C * lane);
  }
  cp_async_commit();
  if (cs_lane) {  // the cos / sin rows wait on the positions: their own group
    if (pos < 0 || pos >= p.max_pos) {
      set_status(p.status, kDevPosRange);
      pos = pos < 0 ? 0 : p.max_pos - 1;
    }
    cp_async16(&ss.cs[lane >> 3][8 * (lane & 7)], p.cos_sin + pos * kRotDim + 8 * (lane & 7));
  }
  cp_async_commit();
  if (FUSED) fused_norm_quant<WFMT>(p, tid, ks, k0, k1, h, x_s, sfb_s, ex1, gin_s, ss.xs, &ss.ex1_bar);
  cp_async_wait<1>();  // weights of batch 0 and the activations
  fence_proxy_async_smem();
  __syncthreads();

  // ------------------------------------------------------------- the MMAs
  for (int c0 = 0, bi = 0; c0 < nch; c0 += kStageChunks, ++bi) {
    if (c0 > 0) {  // a longer K range: the next batch into the freed stages
      issue_weights(c0);
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncthreads();
    }
    if (warp == 4 && lane == 0 && a_tmem) {
      tc_fence_after();
      for (int q = 0; q < 4 * nch; ++q)  // two accumulator chains
        mma_f8_ta(tmem + 16 * (q & 1), tmem + kTaCol + 8 * q,
                  sdesc_sw128(smem_u32(x_s + (q >> 2) * kXChunkBytes)) + 2 * (q & 3), kIdescF8, q >= 2);
      tc_commit(&ss.mma_bar);
    } else if (warp == 4 && lane == 0) {
      tc_fence_after();
      const int n = nch - c0 < kStageChunks ? nch - c0 : kStageChunks;
      for (int j = 0; j < n; ++j) {
        const uint64_t ad = sdesc_sw128(smem_u32(w_s + j * kWChunkBytes));
        const uint64_t bd = sdesc_sw128(smem_u32(x_s + (c0 + j) * kXChunkBytes));
        if (WFMT == 1) {
          tc_cp_sf(tmem + kSfaCol, sdesc_sf(smem_u32(sfa_s + j * kSfAtom)));
          tc_cp_sf(tmem + kSfbCol, sdesc_sf(smem_u32(sfb_s + (c0 + j) * kSfAtom)));
        }
#pragma unroll
        for (int k = 0; k < kChunk / 32; ++k) {
          const uint32_t acc = c0 > 0 || k > 0;
          const uint32_t d = tmem + 16 * j;  // chunk j's accumulator
          // +32 bytes along K inside the swizzle atom: +2 in the 16-byte address field
          if (WFMT == 0) mma_f8(d, ad + 2 * k, bd + 2 * k, kIdescF8, acc);
          else mma_mx(d, ad + 2 * k, bd + 2 * k, kIdescMx | ((uint32_t)k << 4) | ((uint32_t)k << 29),
                      tmem + kSfaCol, tmem + kSfbCol, acc);
        }
      }
      tc_commit(&ss.mma_bar);
    }
    // every thread: the batch's MMAs are done (its stages may be refilled)
    if (!mbar_wait(&ss.mma_bar, bi & 1, p.status, wait_limit(p))) ss.ok = 0;
    __syncthreads();
    if (!ss.ok) break;
  }
  tc_fence_after();
  // ---------------------------------- accumulator -> partial rows of the cluster
  float v[16];
  if (warp < 4) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.f;
    if (ss.ok) {
      // the accumulators used (smem path: accumulator j holds chunks j, j + 3,
      // ...; tensor-memory A: two chains); two loads in flight per wait
      const int nacc = a_tmem ? (nch > 0 ? 2 : 0) : (nch < kStageChunks ? nch : kStageChunks);
      const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
      float u[16];
      if (nacc > 0) tc_ld16(trow, v);
      if (nacc > 1) tc_ld16(trow + 16, u);
      tc_wait_ld();
      if (nacc > 1)
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] += u[i];
      if (nacc > 2) {
        tc_ld16(trow + 32, u);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] += u[i];
      }
    }
  }
  cp_async_wait<0>();  // the cos / sin rows (their own, last group), read by the epilogue
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tc_dealloc(tmem, kTmemCols);
  }
  if (!FUSED) cluster_wait();  // every CTA of the cluster has initialised its barriers
  if (warp < 4) {
    const int r = warp * 32 + lane;  // weight row of the head
#pragma unroll
    for (int m = 0; m < kMaxTok; ++m) {
      if (m < M) {
        float *dst = recv + ((m / C) * C + ks) * kHeadDim + r;
        st_async_b32(mapa(smem_u32(dst), m % C), v[m], mapa(smem_u32(&ss.recv_bar), m % C));
      }
    }
  }
  // ------------------------------------------- head epilogue of token m
  if (warp >= TS) return;
  const int m = ks + C * warp;
  if (m >= M) return;
  if (!mbar_wait_cluster(&ss.recv_bar, 0, p.status, wait_limit(p))) return;
  // testing: a wait that cannot complete (all partials are in, so nothing of
  // the cluster writes here any more), run out like a real one: the row's
  // outputs and done word are skipped and PA_DEV_WAIT_TIMEOUT is raised
  if (p.test_timeout && !mbar_wait(&ss.never_bar, 0, p.status, wait_limit(p))) return;
  const int d0 = 4 * lane;
  float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int q = 0; q < C; ++q) {
    const float4 u = *reinterpret_cast<const float4 *>(recv + (warp * C + q) * kHeadDim + d0);
    y[0] += u.x;
    y[1] += u.y;
    y[2] += u.z;
    y[3] += u.w;
  }
  if (WFMT == 0) {
    const float xs = ss.xs[m];
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = y[i] * xs * ss.wsc[d0 + i];
  }
  HeadCtx hc;
  hc.m = m;
  hc.head = h;
  hc.slot = ss.slot[warp];
  hc.islot = ss.islot[warp];
  hc.cs_row = ss.cs[warp];
  hc.g_q = hc.g_k = hc.g_iq = hc.g_ik = ss.gam;
  head_epilogue<4, CF>(p, hc, y, d0);
}

namespace {

int gv_kc(int H, int C) { return ((H + C - 1) / C + kChunk - 1) / kChunk * kChunk; }
int gv_smem(int C, int kc, int mx) { return gv_layout(C, kc, mx).total + 1024; }  // + alignment slack

// Cluster size usable on the current device: 16 where clusters of 16 CTAs
// with `smem16` bytes of dynamic shared memory can be co-scheduled, else 8.
// Queried once per device and again only for a larger shared-memory size;
// the attributes it sets stay set.
template <int WFMT>
int pick_cluster(int smem16) {
  struct Entry {
    int c, smem;
  };
  static Entry cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
  if (cached[dev].c && cached[dev].smem >= smem16) return cached[dev].c;
  int c = 8;
  const void *k16[4] = {reinterpret_cast<const void *>(pa_skinny_proj_kernel<WFMT, 16, false, 0>),
                        reinterpret_cast<const void *>(pa_skinny_proj_kernel<WFMT, 16, true, 0>),
                        reinterpret_cast<const void *>(pa_skinny_proj_kernel<WFMT, 16, false, 1>),
                        reinterpret_cast<const void *>(pa_skinny_proj_kernel<WFMT, 16, true, 1>)};
  bool failed = false;
  for (const void *k : k16) {
    if (!failed) failed = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess;
    if (!failed) failed = ensure_smem_attr(k, smem16) != cudaSuccess;
  }
  if (!failed) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(16 * 64);
    cfg.blockDim = dim3(kGvThreads);
    cfg.dynamicSmemBytes = smem16;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    failed = cudaOccupancyMaxActiveClusters(&n, k16[1], &cfg) != cudaSuccess;
    if (!failed && n >= 1) c = 16;
  }
  if (failed) cudaGetLastError();  // a refused attribute or query only means: clusters of 8
  cached[dev] = Entry{c, smem16};
  return c;
}

template <int WFMT, int C, bool FUSED, int CF>
cudaError_t launch_c(const Params &p, bool pdl, cudaStream_t stream) {
  const int kc = gv_kc(p.H, C);
  const int smem = gv_smem(C, kc, WFMT);
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(pa_skinny_proj_kernel<WFMT, C, FUSED, CF>), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(p.n_heads * C);
  cfg.blockDim = dim3(kGvThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, pa_skinny_proj_kernel<WFMT, C, FUSED, CF>, p, kc, (int)pdl);
}

template <int WFMT>
bool fused_ok(int H) {
  return gv_kc(H, 16) <= kFusedMaxKc && pick_cluster<WFMT>(gv_smem(16, gv_kc(H, 16), WFMT)) == 16;
}

template <int WFMT, int CF>
cudaError_t launch_t(const Params &p, bool fused, bool pdl, cudaStream_t stream) {
  if (fused) return launch_c<WFMT, 16, true, CF>(p, pdl, stream);
  if (pick_cluster<WFMT>(gv_smem(16, gv_kc(p.H, 16), WFMT)) == 16) return launch_c<WFMT, 16, false, CF>(p, pdl, stream);
  return launch_c<WFMT, 8, false, CF>(p, pdl, stream);
}

}  // namespace

bool gemv_fuses_prologue(int H, int weight_fmt) { return weight_fmt == 0 ? fused_ok<0>(H) : fused_ok<1>(H); }

int gemv_regular_clusters(int weight_fmt, int H) {
  const int smem = gv_smem(16, gv_kc(H, 16), weight_fmt);
  if ((weight_fmt == 0 ? pick_cluster<0>(smem) : pick_cluster<1>(smem)) != 16) return 0;
  const void *k = weight_fmt == 0 ? reinterpret_cast<const void *>(pa_skinny_proj_kernel<0, 16, false, 0>)
                                  : reinterpret_cast<const void *>(pa_skinny_proj_kernel<1, 16, false, 0>);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(16 * 64);
  cfg.blockDim = dim3(kGvThreads);
  cfg.dynamicSmemBytes = smem;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 16;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_gemv(const Params &p, bool fused, bool pdl, cudaStream_t stream) {
  if (p.cache_fmt == 0)
    return p.weight_fmt == 0 ? launch_t<0, 0>(p, fused, pdl, stream) : launch_t<1, 0>(p, fused, pdl, stream);
  return p.weight_fmt == 0 ? launch_t<0, 1>(p, fused, pdl, stream) : launch_t<1, 1>(p, fused, pdl, stream);
}

}  // namespace pa
