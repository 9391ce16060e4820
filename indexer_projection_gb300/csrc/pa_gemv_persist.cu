// Skinny-M path for many heads: the GEMV of pa_gemv.cu, persistent.
//
// With more heads than clusters of 16 CTAs fit on the device at once (77
// heads at nkv = 4), the one-cluster-a-head grid runs in waves, and the
// weight stream stops between them while each wave's CTAs start up, reduce
// and run their epilogues.  Here G clusters (as many as are resident at once)
// each take heads c, c + G, c + 2G, ...; a CTA keeps its K range of the
// activations staged once and walks its heads through rings, so the weight
// stream never waits for one head's reduction or epilogue:
//   - one thread copies a head's weight slice (128 rows x this K range,
//     128-byte swizzled TMA boxes, and the MXFP8 scale atoms) into stage
//     i % kPgS once the MMAs of head i - kPgS have read it;
//   - one thread issues head i's MMAs (tcgen05, m128 n16 k32, tokens as the
//     16 columns, the whole K range into one accumulator) into tensor-memory
//     accumulator i % kPgS once the readers of head i - kPgS have drained it;
//   - warps 0-3 read the accumulator (thread = weight row) and, once every
//     token's owner has read head i - 2's partials out of receive buffer
//     i % 2, send token m's partial row to cluster CTA m with byte-counted
//     st.async;
//   - in the CTA that owns token m (m < M <= 16), warps 6 and 7 take the even
//     and the odd heads: wait for the 16 partials in their receive buffer,
//     sum them, re-arm the buffer's barrier, tell every CTA of the cluster the
//     buffer is free (remote mbarrier arrivals) and run the head epilogue
//     (gamma from shared memory, the next head's per-channel scales already
//     loaded), so an epilogue may take two heads' time; warp 8 loads the
//     token's slots and cos / sin row meanwhile.
// Only the first head's weights are requested before the wait on the
// previous kernel; the activations are requested next and the other stages
// after them, since loads queue behind the weight stream.  The remote
// arrivals are relaxed (a release there waited for the stream too).
// The arithmetic per head is the regular kernel's (pa_gemv.cu) with the
// weights read from shared memory (MXFP8: the same MMAs, bit for bit; the
// per-channel format's sums can differ in the last bits from the regular
// kernel's two tensor-memory chains).  K <= 16 x 384 (three 128-byte chunks
// a range).
// Every wait is bounded; the CTAs of a cluster leave together (a cluster
// barrier), so no CTA exits while another may still write to it.
#include "../../include/pre_attn.h"
#include "pa_device.cuh"
#include "pa_launch.h"
#include "pa_tc.cuh"
#include "pa_tma.h"

namespace pa {
namespace {

constexpr int kPgThreads = 288;
constexpr int kPgC = 16;                    // CTAs a cluster = K ranges
constexpr int kPgS = 4;                     // weight stages = tensor-memory accumulators
constexpr int kPgChunk = 128;               // K bytes of a swizzle-atom column (4 MMAs)
constexpr int kPgMaxCh = 3;                 // chunks a K range
constexpr int kPgW = kHeadDim * kPgChunk;   // 16 KB: a chunk of a head's weight slice
constexpr int kPgX = 16 * kPgChunk;         // 2 KB: a chunk of the 16 token rows
constexpr int kPgSf = 512;                  // F8_128x4 scale atom
constexpr int kPgMaxTok = 16;
constexpr int kPgRecv = kPgC * kHeadDim * 4;  // 8 KB: the 16 partial rows of the owned token
constexpr uint32_t kPgTmemCols = 128;       // accumulator b at column 16 b, scale atoms after them
constexpr int kPgSfaCol = 16 * kPgS, kPgSfbCol = 16 * kPgS + 4;
constexpr uint32_t kPgIdescF8 = idesc_f8(128, 16);
constexpr uint32_t kPgIdescMx = idesc_mx(128, 16);
static_assert(kPgSfbCol + 4 <= (int)kPgTmemCols, "tensor-memory columns");

// dynamic shared memory, from a 1024-byte aligned base
constexpr int kOffW = 0;                                  // [kPgS][3] weight chunks
constexpr int kOffX = kOffW + kPgS * kPgMaxCh * kPgW;     // [3] activation chunks
constexpr int kOffSfa = kOffX + kPgMaxCh * kPgX;          // [kPgS][3] weight scale atoms (MXFP8)
constexpr int kOffSfb = kOffSfa + kPgS * kPgMaxCh * kPgSf;  // [3] activation scale atoms (MXFP8)
constexpr int kOffRecv = kOffSfb + kPgMaxCh * kPgSf;      // [2][16 K ranges][128] f32 partial rows
constexpr int kPgSmem = kOffRecv + 2 * kPgRecv + 1024;    // + alignment slack

struct alignas(16) PgStatic {  // cs and gam are 16-byte cp.async destinations
  __nv_bfloat16 cs[kRotDim];        // cos / sin row of the owned token
  __nv_bfloat16 gam[4][kHeadDim];   // gamma of q, k, index_q, index_k heads
  float xs[kPgMaxTok];              // per-token activation scales (per-channel format)
  int64_t slot, islot;              // the owned token's cache slots
  uint64_t w_full[kPgS], w_empty[kPgS], acc_full[kPgS], acc_empty[kPgS];
  uint64_t recv_bar[2], recv_free[2], tok_ready, never_bar, drain;
  uint32_t tmem;
};

__device__ __forceinline__ int pg_swz(int r, int c) { return (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ void pg_tma(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Remote arrival without release semantics.  A release here waits until
// this SM's earlier memory traffic is performed, which behind the weight
// stream took 1-2 us a head.  What it must order is the arriving warp's
// reads of the receive buffer before the senders overwrite it: the sums
// passed in consume every one of those reads, and a warp issues in order, so
// the arrival cannot issue before the reads have returned.
__device__ __forceinline__ void pg_arrive_after(uint32_t caddr, const float (&y)[4]) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr), "f"(y[0]), "f"(y[1]),
               "f"(y[2]), "f"(y[3])
               : "memory");
}

__device__ __forceinline__ void pg_st_async(uint32_t caddr, float v, uint32_t cbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(caddr),
               "r"(__float_as_uint(v)), "r"(cbar)
               : "memory");
}

template <int WFMT, int CF>
__global__ void __launch_bounds__(kPgThreads, 1)
    pa_skinny_persist_kernel(const __grid_constant__ CUtensorMap tmW, Params p, int kc, int use_pdl) {
  extern __shared__ uint8_t dsm_raw[];
  uint8_t *dsm = dsm_raw + ((1024 - (smem_u32(dsm_raw) & 1023)) & 1023);
  __shared__ PgStatic ss;
  uint8_t *w_s = dsm + kOffW, *x_s = dsm + kOffX, *sfa_s = dsm + kOffSfa, *sfb_s = dsm + kOffSfb;
  float *recv = reinterpret_cast<float *>(dsm + kOffRecv);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = p.H, M = p.M, ksf = K >> 5;
  const int ks = (int)cta_rank();  // this CTA's K range, and the token it finishes
  const int cid = blockIdx.x / kPgC, G = gridDim.x / kPgC;
  const int k0 = ks * kc, k1 = k0 + kc < K ? k0 + kc : K;
  const int nch = k1 > k0 ? (k1 - k0) / kPgChunk : 0;
  const int nh = cid < p.n_heads ? (p.n_heads - cid + G - 1) / G : 0;  // heads of this cluster
  const bool owner = ks < M;
  const int n_owners = M < kPgC ? M : kPgC;
  const uint64_t lim = wait_limit(p);
  const uint32_t wbytes = (uint32_t)nch * (kPgW + (WFMT == 1 ? kPgSf : 0));

  if (tid == 0) {
    for (int b = 0; b < kPgS; ++b) {
      mbar_init(&ss.w_full[b], 1);
      mbar_init(&ss.w_empty[b], 1);
      mbar_init(&ss.acc_full[b], 1);
      mbar_init(&ss.acc_empty[b], 4);  // the four reader warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ss.recv_bar[b], 1);
      // heads 0 and 1: 16 partial rows each
      if (owner && b < nh) mbar_expect_tx(&ss.recv_bar[b], kPgRecv);
      mbar_init(&ss.recv_free[b], n_owners);  // every owner, once a head
    }
    mbar_init(&ss.tok_ready, 1);
    mbar_init(&ss.never_bar, 1);
    mbar_init(&ss.drain, 1);
    fence_mbar_init();
  }
  if (warp == 4) tc_alloc(&ss.tmem, kPgTmemCols);
  cluster_arrive_relaxed();  // matched by cluster_wait() before the first remote operation

  // head i's weight slice into stage i % kPgS (the producer thread)
  auto issue_head = [&](int i) {
    const int b = i % kPgS, h = cid + i * G;
    mbar_expect_tx(&ss.w_full[b], wbytes);
    for (int j = 0; j < nch; ++j) {
      pg_tma(w_s + (b * kPgMaxCh + j) * kPgW, &tmW, k0 + j * kPgChunk, h * kHeadDim, &ss.w_full[b]);
      if (WFMT == 1)
        bulk_g2s(sfa_s + (b * kPgMaxCh + j) * kPgSf,
                 p.wsf + ((int64_t)h * (ksf >> 2) + (k0 / kPgChunk) + j) * kPgSf, kPgSf, &ss.w_full[b]);
    }
  };
  __syncthreads();  // the barriers are initialised
  // the first stage's weights before the wait (model constants); the other
  // stages are requested after the activations, which would otherwise queue
  // behind them (the MMAs wait for the activations, the stream for the MMAs)
  if (warp == 5 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
    if (nh > 0) issue_head(0);
  }
  if (warp == 6) {  // the gammas (model constants) before the wait
    const __nv_bfloat16 *src = lane < 16 ? (lane < 8 ? p.g_q : p.g_k) : (lane < 24 ? p.g_iq : p.g_ik);
    cp_async16(&ss.gam[lane >> 3][16 * (lane & 7)], src + 16 * (lane & 7));
    cp_async16(&ss.gam[lane >> 3][16 * (lane & 7) + 8], src + 16 * (lane & 7) + 8);
  }
  if (warp == 8 && lane == 0 && owner) {  // the owned token's inputs: a hint before the wait
    prefetch_l2(p.pos + ks);
    prefetch_l2(p.slot + ks);
    prefetch_l2(p.islot + ks);
  }
  if (use_pdl) {
    pdl_trigger();
    pdl_wait();
  }
  // ------------------------------------------ activations and per-token data (once)
  for (int i = tid; i < nch * 16 * 8; i += kPgThreads) {
    const int j = i >> 7, rc = i & 127, r = rc >> 3, c = rc & 7;
    uint8_t *dst = x_s + j * kPgX + pg_swz(r, c);
    if (r < M) cp_async16(dst, p.xq + (int64_t)r * K + k0 + j * kPgChunk + 16 * c);
    else *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (WFMT == 1)
    for (int i = tid; i < nch * (kPgSf / 16); i += kPgThreads) {
      const int j = i / (kPgSf / 16), c = i - j * (kPgSf / 16);
      cp_async16(sfb_s + j * kPgSf + 16 * c, p.xsf + ((int64_t)(k0 / kPgChunk) + j) * kPgSf + 16 * c);
    }
  if (WFMT == 0 && tid < M) cp_async4(&ss.xs[tid], p.x_scale + tid);
  cp_async_commit();
  if (warp == 5 && lane == 0)
    for (int i = 1; i < nh && i < kPgS; ++i) issue_head(i);
  cp_async_wait<0>();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ss.tmem;
  cluster_wait();  // every CTA of the cluster has initialised its barriers

  if (warp == 5) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int i = kPgS;
      for (; i < nh; ++i) {
        const int b = i % kPgS;
        if (!mbar_wait(&ss.w_empty[b], ((uint32_t)(i / kPgS) & 1) ^ 1, p.status, lim)) break;
        issue_head(i);
      }
      if (i < nh)  // a wait ran out: the copies in flight land before the CTA exits
        for (int k = i - 1; k >= 0 && k >= i - kPgS; --k)
          mbar_wait(&ss.w_full[k % kPgS], (uint32_t)(k / kPgS) & 1, p.status, lim);
    }
  } else if (warp == 4) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int i = 0; i < nh && ok; ++i) {
        const int b = i % kPgS;
        const uint32_t ph = (uint32_t)(i / kPgS) & 1;
        if (!mbar_wait(&ss.w_full[b], ph, p.status, lim) || !mbar_wait(&ss.acc_empty[b], ph ^ 1, p.status, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + 16 * b;  // the head's accumulator: its whole K range
        for (int j = 0; j < nch; ++j) {
          const uint64_t ad = sdesc_sw128(smem_u32(w_s + (b * kPgMaxCh + j) * kPgW));
          const uint64_t bd = sdesc_sw128(smem_u32(x_s + j * kPgX));
          if (WFMT == 1) {
            tc_cp_sf(tmem + kPgSfaCol, sdesc_sf(smem_u32(sfa_s + (b * kPgMaxCh + j) * kPgSf)));
            tc_cp_sf(tmem + kPgSfbCol, sdesc_sf(smem_u32(sfb_s + j * kPgSf)));
          }
#pragma unroll
          for (int k = 0; k < kPgChunk / 32; ++k) {
            // +32 bytes along K inside the swizzle atom: +2 in the 16-byte address field
            if (WFMT == 0) mma_f8(d, ad + 2 * k, bd + 2 * k, kPgIdescF8, (j | k) != 0);
            else mma_mx(d, ad + 2 * k, bd + 2 * k, kPgIdescMx | ((uint32_t)k << 4) | ((uint32_t)k << 29),
                        tmem + kPgSfaCol, tmem + kPgSfbCol, (j | k) != 0);
          }
        }
        tc_commit(&ss.w_empty[b]);   // the weight stage is free once these MMAs have read it
        tc_commit(&ss.acc_full[b]);
      }
      if (!ok) {  // the MMAs issued complete before the tensor memory is freed
        tc_commit(&ss.drain);
        mbar_wait(&ss.drain, 0, p.status, lim);
      }
    }
  } else if (warp < 4) {
    // ------------------------------------- accumulator -> partial rows of the owners
    const int r = warp * 32 + lane;  // weight row of the head
    for (int i = 0; i < nh; ++i) {
      const int b = i % kPgS, rb = i & 1;
      float v[16];
      const bool got = mbar_wait(&ss.acc_full[b], (uint32_t)(i / kPgS) & 1, p.status, lim);
      if (__any_sync(0xffffffffu, !got)) break;
      tc_fence_after();
      if (nch > 0) {
        tc_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 16 * b, v);
        tc_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0.f;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ss.acc_empty[b]);
      // every owner has read head i - 2's partials out of receive buffer rb
      const bool fr =
          i < 2 || mbar_wait_cluster(&ss.recv_free[rb], ((uint32_t)(i >> 1) & 1) ^ 1, p.status, lim);
      if (__any_sync(0xffffffffu, !fr)) break;
      const uint32_t dst = smem_u32(recv + rb * (kPgRecv / 4) + ks * kHeadDim + r);
      const uint32_t bar = smem_u32(&ss.recv_bar[rb]);
#pragma unroll
      for (int m = 0; m < kPgMaxTok; ++m)
        if (m < M) pg_st_async(mapa(dst, m), v[m], mapa(bar, m));
    }
  } else if ((warp == 6 || warp == 7) && owner) {
    // --------------------------------- head epilogues of token ks (even / odd heads)
    const int m = ks, d0 = 4 * lane, e = warp - 6;
    bool tok = false;
    float4 wsc_next = make_float4(0.f, 0.f, 0.f, 0.f);
    if (WFMT == 0 && e < nh)
      wsc_next = __ldg(reinterpret_cast<const float4 *>(p.w_scale + (int64_t)(cid + e * G) * kHeadDim + d0));
    for (int i = e; i < nh; i += 2) {
      const int h = cid + i * G, rb = i & 1;
      const float4 wsc = wsc_next;
      if (WFMT == 0 && i + 2 < nh)  // in flight while this head is received and finished
        wsc_next = __ldg(reinterpret_cast<const float4 *>(p.w_scale + (int64_t)(h + 2 * G) * kHeadDim + d0));
      if (!mbar_wait_cluster(&ss.recv_bar[rb], (uint32_t)(i >> 1) & 1, p.status, lim)) break;
      const float *rv = recv + rb * (kPgRecv / 4);
      float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < kPgC; ++q) {
        const float4 t = *reinterpret_cast<const float4 *>(rv + q * kHeadDim + d0);
        y[0] += t.x;
        y[1] += t.y;
        y[2] += t.z;
        y[3] += t.w;
      }
      // the buffer is read: re-armed for head i + 2, and free for every CTA
      __syncwarp();
      if (i + 2 < nh) {
        if (lane == 0) mbar_expect_tx(&ss.recv_bar[rb], kPgRecv);
        __syncwarp();
        if (lane < kPgC) pg_arrive_after(mapa(smem_u32(&ss.recv_free[rb]), lane), y);
      }
      if (!tok) {  // the token's slots and cos / sin row (warp 8)
        if (!mbar_wait(&ss.tok_ready, 0, p.status, lim)) break;
        tok = true;
      }
      // testing: a wait that cannot complete, run out like a real one: the
      // row's outputs are skipped and PA_DEV_WAIT_TIMEOUT is raised
      if (p.test_timeout && !mbar_wait(&ss.never_bar, 0, p.status, lim)) continue;
      if (WFMT == 0) {
        const float xs = ss.xs[m];
        y[0] = y[0] * xs * wsc.x;
        y[1] = y[1] * xs * wsc.y;
        y[2] = y[2] * xs * wsc.z;
        y[3] = y[3] * xs * wsc.w;
      }
      HeadCtx hc;
      hc.m = m;
      hc.head = h;
      hc.slot = ss.slot;
      hc.islot = ss.islot;
      hc.cs_row = ss.cs;
      hc.g_q = ss.gam[0];
      hc.g_k = ss.gam[1];
      hc.g_iq = ss.gam[2];
      hc.g_ik = ss.gam[3];
      head_epilogue<4, CF>(p, hc, y, d0);
    }
  } else if (warp == 8 && owner) {
    // ------------------- the owned token's slots and cos / sin row, off the
    // path to the first MMA (a dependent pair of loads behind the weights)
    if (lane == 0) {
      cp_async8(&ss.slot, p.slot + ks);
      cp_async8(&ss.islot, p.islot + ks);
    }
    if (lane < 8) {
      int64_t pos = ld_i64(p.pos + ks);
      if (pos < 0 || pos >= p.max_pos) {
        if (lane == 0) set_status(p.status, kDevPosRange);
        pos = pos < 0 ? 0 : p.max_pos - 1;
      }
      cp_async16(&ss.cs[8 * lane], p.cos_sin + pos * kRotDim + 8 * lane);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ss.tok_ready);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tc_dealloc(tmem, kPgTmemCols);
  }
  cluster_sync();  // no CTA leaves while another may still signal or write to it
}

struct PersistInfo {
  int clusters;  // resident clusters of the persistent kernel (0: not launchable)
  int regular;   // resident clusters of 16 of the regular kernel
};

template <int WFMT>
PersistInfo persist_info(int H) {
  static PersistInfo cached[64][2] = {};
  static bool done[64][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PersistInfo{0, 0};
  if (done[dev][WFMT]) return cached[dev][WFMT];
  PersistInfo r{0, 0};
  auto clusters_of = [](const void *k, int smem) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(kPgC * 64);
    cfg.blockDim = dim3(kPgThreads);
    cfg.dynamicSmemBytes = smem;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPgC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
        ensure_smem_attr(k, smem) != cudaSuccess || cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess)
      n = 0;
    return n;
  };
  r.clusters = clusters_of(reinterpret_cast<const void *>(pa_skinny_persist_kernel<WFMT, 0>), kPgSmem);
  r.regular = gemv_regular_clusters(WFMT, H);
  cudaGetLastError();  // a refused query only means: not used
  for (int cf = 0; cf < 2; ++cf) {
    const void *k = cf ? reinterpret_cast<const void *>(pa_skinny_persist_kernel<WFMT, 1>)
                       : reinterpret_cast<const void *>(pa_skinny_persist_kernel<WFMT, 0>);
    if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
        ensure_smem_attr(k, kPgSmem) != cudaSuccess)
      r.clusters = 0;
  }
  cudaGetLastError();
  cached[dev][WFMT] = r;
  done[dev][WFMT] = true;
  return r;
}

template <int WFMT, int CF>
cudaError_t launch_p(const Params &p, int clusters, bool pdl, cudaStream_t stream) {
  CUtensorMap tmW;
  if (!map_rows_sw128(&tmW, p.w, (uint64_t)p.N, (uint64_t)p.H, kPgChunk, kHeadDim)) return cudaErrorInvalidValue;
  const int kc = ((p.H + kPgC - 1) / kPgC + kPgChunk - 1) / kPgChunk * kPgChunk;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(clusters * kPgC);
  cfg.blockDim = dim3(kPgThreads);
  cfg.dynamicSmemBytes = kPgSmem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPgC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, pa_skinny_persist_kernel<WFMT, CF>, tmW, p, kc, (int)pdl);
}

}  // namespace

int gemv_persist_clusters(int n_heads, int H, int weight_fmt, bool force) {
  if (H > kPgC * kPgMaxCh * kPgChunk || H % kPgChunk) return 0;
  const PersistInfo r = weight_fmt == 0 ? persist_info<0>(H) : persist_info<1>(H);
  if (r.clusters < 1) return 0;
  // with a few heads a resident cluster the regular grid, whose clusters
  // start and drain independently, is faster (measured with 7 resident
  // clusters: 20 heads, 7.2 vs 9.3 us a step); from about four on (39 heads:
  // 11.4 vs 12.2 us; 77 heads: 15.0 vs 21.1 us) this kernel is
  if (!force && (n_heads <= r.regular || n_heads <= 4 * r.clusters)) return 0;
  return n_heads < r.clusters ? n_heads : r.clusters;
}

cudaError_t launch_gemv_persist(const Params &p, int clusters, bool pdl, cudaStream_t stream) {
  if (p.cache_fmt == 0)
    return p.weight_fmt == 0 ? launch_p<0, 0>(p, clusters, pdl, stream) : launch_p<1, 0>(p, clusters, pdl, stream);
  return p.weight_fmt == 0 ? launch_p<0, 1>(p, clusters, pdl, stream) : launch_p<1, 1>(p, clusters, pdl, stream);
}

}  // namespace pa
