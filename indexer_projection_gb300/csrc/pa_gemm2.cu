// Tensor-core path on CTA pairs (cta_group::2): a persistent tcgen05 GEMM
// whose 2-CTA cluster computes a 256 x 256 output tile per step of K, with
// the per-head epilogue fused behind the TMEM accumulator.
//
//   pair      CTA r of the cluster owns token rows (2*mp + r)*128 .. +128 and
//             loads the B rows n*256 + r*128 .. +128 (half of the tile's N);
//             one m256 n256 k32 MMA, issued by CTA 0, reads both CTAs' A and
//             B ("vllm.models.minimax_m3.nvidia.ops.qkv_index_fused_epilogue",
//             QkvIndexFusedEpilogueKernel, cta_group=2).  Per FLOP each SM
//             reads half the shared-memory operand bytes of a 128 x 128 tile,
//             and the ring covers twice the load latency.
//   TMEM      each CTA: a 256-column accumulator (its 128 rows x the two
//             heads of the tile) and 12 scale-factor columns; the epilogue
//             drains it into registers and releases it at once, so the next
//             tile's MMAs overlap the epilogue's arithmetic and stores.
//   warps     0-7 epilogue (warpgroup g takes head 2n + g, a thread a row),
//             8 TMA producer, 9 TMEM allocator + MMA issuer (CTA 0 issues).
//   loads     A, B: 128 x 128-byte TMA tiles, 128B swizzle; MXFP8 scales:
//             the F8_128x4 atoms (512 B) by TMA, SFA for the CTA's own rows,
//             SFB for both halves of N (each CTA needs all 256 columns'
//             scales; no multicast).  Every load of both CTAs completes on
//             CTA 0's stage barrier (TMA .cta_group::2), which CTA 0 alone
//             arms with both CTAs' byte count.
//   odd head count: the last N tile's second head is zero-filled by TMA and
//             never stored.
// Every mbarrier wait is bounded (about a second); a timeout raises
// PA_DEV_WAIT_TIMEOUT and the kernel still reaches its final cluster barrier
// and frees its TMEM.
#include "pa_device.cuh"
#include "pa_launch.h"
#include "pa_tc.cuh"
#include "pa_tma.h"

namespace pa {
namespace g2 {

constexpr int kBM = 128, kBN = 256, kBK = 128;  // per CTA: 128 rows x the pair's 256 columns
constexpr int kStages = 6;
constexpr int kTile = 128 * kBK;  // 16 KB: A tile, or this CTA's half of B
constexpr int kSf = 512;          // one F8_128x4 atom
constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int kTmemCols = 512;
constexpr int kSfaCol = 256, kSfbCol = 260;

struct Smem {  // offsets from the 1024-aligned base
  static constexpr int a = 0;
  static constexpr int b = a + kStages * kTile;
  static constexpr int sfa = b + kStages * kTile;
  static constexpr int sfb = sfa + kStages * 1024;          // 1024-aligned slots
  static constexpr int bars = sfb + kStages * 1024;          // full[S], empty[S], tfull, tempty, never, drain
  static constexpr int tmem_addr = bars + (2 * kStages + 4) * 8;
  static constexpr int ok = tmem_addr + 8;                   // 2 x int: tile verdicts (+ 8 bytes: wscale 16-aligned)
  static constexpr int wscale = ok + 16;                     // [2 parity][2 heads][128] f32
  static constexpr int total = wscale + 2 * 2 * 128 * 4;
};
constexpr int kSmemBytes = Smem::total + 1024;

// ------------------------------------------------------------- cluster PTX
// 2-D TMA load into this CTA's shared memory, completing on a barrier that
// may sit in the peer CTA (cta_group::2).
__device__ __forceinline__ void tma_2d_pair(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t cbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cbar)
      : "memory");
}

// M = 256 (the pair), N = 256, A and B E4M3, K-major.
constexpr uint32_t kIdescF8 = idesc_f8(256, 256);
constexpr uint32_t kIdescMx = idesc_mx(256, 256);

__device__ __forceinline__ void mma_f8_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{.reg .pred p; setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_mx_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                       uint32_t acc) {
  asm volatile(
      "{.reg .pred p; setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tc_cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// arrive once on the barrier at this offset in both CTAs of the pair
__device__ __forceinline__ void tc_commit_pair(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

// Tile raster (chosen on the host, the same for every CTA): tiles are
// numbered in groups of group_m m-pairs, the m-pair running fastest inside a
// group, then the n tile ("vllm.models.minimax_m3.nvidia.ops.
// qkv_index_fused_epilogue", QkvIndexFusedEpilogueKernel.tile_coords /
// _group_m).  The clusters of one wave then share a few weight tiles, and a
// group's activations stay in L2 while it walks every weight tile: the
// weights are read from HBM about once per group rather than once per wave.
struct Sched {
  int m_pairs, n_tiles, ksteps, group_m;
};

__device__ __forceinline__ void tile_coords(const Sched &s, int tile, int &mp, int &nt) {
  const int per = s.group_m * s.n_tiles;
  const int g = tile / per, idx = tile - g * per;
  const int gm = s.m_pairs - g * s.group_m < s.group_m ? s.m_pairs - g * s.group_m : s.group_m;
  nt = idx / gm;
  mp = g * s.group_m + (idx - nt * gm);
}
// The cluster's tiles, in order: tile c, c + C, ..., K steps [0, ksteps)
// each, as a running count of K steps.  The three roles (TMA producer, MMA
// issuer, epilogue) walk the same sequence.  (Written this way, rather than
// as a plain loop over tiles, the kernel compiled to fewer epilogue spills
// and ran ~5% faster on prefill.)
struct Segs {
  int tile, ks0, ks1;
  int u, u1, ksteps, step;
  __device__ Segs(const Sched &s, int c, int C) : ksteps(s.ksteps) {
    u = c * ksteps;
    u1 = s.m_pairs * s.n_tiles * ksteps;
    step = C * ksteps;
    set();
  }
  __device__ bool valid() const { return u < u1; }
  __device__ void set() {
    tile = u / ksteps;
    ks0 = u - tile * ksteps;
    ks1 = ksteps;
  }
  __device__ void next() {
    u += step;
    set();
  }
};
template <int WFMT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    pa_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB, Params p,
                 Sched sc, int use_pdl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Smem::bars);
  uint64_t *empty = full + kStages;
  uint64_t *tfull = empty + kStages;
  uint64_t *tempty = tfull + 1;
  uint64_t *never = tempty + 1;  // testing: nothing arrives on it
  uint64_t *drain = never + 1;   // the MMA issuer's last commit on an abnormal exit
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Smem::tmem_addr);
  volatile int *ok_s = reinterpret_cast<volatile int *>(smem + Smem::ok);
  float *ws_s = reinterpret_cast<float *>(smem + Smem::wscale);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cta_rank();
  const int M = p.M, K = p.H;
  const int cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);   // CTA 0's expect_tx arrival, for both CTAs' bytes
      mbar_init(&empty[s], 1);  // the MMA's commit
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 4);  // one arrival per epilogue warpgroup of each CTA
    mbar_init(never, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (use_pdl) {
    pdl_trigger();
    pdl_wait();
  }
  const uint32_t full0 = mapa(smem_u32(full), 0);      // stage barriers of CTA 0
  const uint32_t tempty0 = mapa(smem_u32(tempty), 0);  // accumulator-free barrier of CTA 0

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t tx = 2 * kTile + (WFMT == 1 ? 3 * kSf : 0);
      bool ok = true;
      int last_ph[kStages];  // phase each stage was last armed with (-1: never)
#pragma unroll
      for (int i = 0; i < kStages; ++i) last_ph[i] = -1;
      for (Segs sg(sc, cluster, clusters); sg.valid() && ok; sg.next()) {
        int mp, nt;
        tile_coords(sc, sg.tile, mp, nt);
        const int m_tile = 2 * mp + (int)rank;
        for (int ks = sg.ks0; ks < sg.ks1; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.status, wait_limit(p))) {
            ok = false;
            break;
          }
          last_ph[stage] = (int)phase;
          const uint32_t fb = full0 + stage * 8;
          // CTA 0 expects both CTAs' bytes on its own barrier (a local
          // arrival); CTA 1's loads just complete their bytes there.  A
          // remote arrival per stage would put a cluster-scope release on
          // CTA 1's load path every k-step.
          if (rank == 0) mbar_expect_tx(&full[stage], 2 * tx);
          tma_2d_pair(smem_u32(smem + Smem::a + stage * kTile), &tmA, ks * kBK, m_tile * kBM, fb);
          tma_2d_pair(smem_u32(smem + Smem::b + stage * kTile), &tmB, ks * kBK, nt * kBN + (int)rank * 128, fb);
          if (WFMT == 1) {
            tma_2d_pair(smem_u32(smem + Smem::sfa + stage * 1024), &tmSFA, ks * 64, m_tile, fb);
            tma_2d_pair(smem_u32(smem + Smem::sfb + stage * 1024), &tmSFB, ks * 64, 2 * nt, fb);
            tma_2d_pair(smem_u32(smem + Smem::sfb + stage * 1024 + kSf), &tmSFB, ks * 64, 2 * nt + 1, fb);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // a wait ran out: the copies already issued (both CTAs' bytes count on
      // CTA 0's stage barriers) land before the pair passes its final cluster
      // barrier
      if (!ok && rank == 0)
#pragma unroll
        for (int i = 0; i < kStages; ++i)
          if (last_ph[i] >= 0) mbar_wait(&full[i], (uint32_t)last_ph[i], p.status, wait_limit(p));
    }
  } else if (warp == 9) {
    // -------------------------------------------------- MMA issuer (CTA 0)
    if (rank == 0 && lane == 0) {
      int stage = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true;
      const uint32_t a0 = smem_u32(smem + Smem::a), b0 = smem_u32(smem + Smem::b);
      const uint32_t sfa0 = smem_u32(smem + Smem::sfa), sfb0 = smem_u32(smem + Smem::sfb);
      for (Segs sg(sc, cluster, clusters); sg.valid() && ok; sg.next()) {
        if (!mbar_wait(tempty, aphase ^ 1, p.status, wait_limit(p))) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = sg.ks0; ks < sg.ks1; ++ks) {
          if (!mbar_wait(&full[stage], phase, p.status, wait_limit(p))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(a0 + stage * kTile), bd = sdesc_sw128(b0 + stage * kTile);
          if (WFMT == 1) {
            tc_cp_sf_pair(tmem + kSfaCol, sdesc_sf(sfa0 + stage * 1024));
            tc_cp_sf_pair(tmem + kSfbCol, sdesc_sf(sfb0 + stage * 1024));
            tc_cp_sf_pair(tmem + kSfbCol + 4, sdesc_sf(sfb0 + stage * 1024 + kSf));
          }
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k) {
            const uint32_t acc = ks > sg.ks0 || k > 0;
            if (WFMT == 0) {
              mma_f8_pair(tmem, ad + 2 * k, bd + 2 * k, kIdescF8, acc);
            } else {
              const uint32_t idesc = kIdescMx | ((uint32_t)k << 4) | ((uint32_t)k << 29);
              mma_mx_pair(tmem, ad + 2 * k, bd + 2 * k, idesc, tmem + kSfaCol, tmem + kSfbCol, acc);
            }
          }
          tc_commit_pair(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        tc_commit_pair(tfull);
        aphase ^= 1;
      }
      if (!ok) {  // a wait ran out: the MMAs already issued complete before the TMEM is freed
        tc_commit_pair(drain);
        mbar_wait(drain, 0, p.status, wait_limit(p));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wg = warp >> 2;              // head of the tile
    const int row = (warp & 3) * 32 + lane;  // TMEM lane and tile row
    const int erow = wg * 128 + row;       // 0..255 across both warpgroups
    uint32_t aphase = 0;
    int it = 0;
    for (Segs sg(sc, cluster, clusters); sg.valid(); sg.next(), ++it) {
      int mp, nt;
      tile_coords(sc, sg.tile, mp, nt);
      const int head = 2 * nt + wg;
      // the row's position, slots and scale, and its cos / sin line, fetched
      // while the tile's MMAs run (they do not depend on them)
      const int m = (2 * mp + (int)rank) * kBM + row;
      const bool live = m < M && head < p.n_heads;
      int64_t pos = 0, slot = -1, islot = -1;
      float xs = 1.0f;
      if (live) {
        pos = load_pos(p, m);
        slot = ld_i64(p.slot + m);
        islot = ld_i64(p.islot + m);
        if (WFMT == 0) xs = __ldcg(p.x_scale + m);
        asm volatile("prefetch.global.L1 [%0];" ::"l"(p.cos_sin + pos * kRotDim));
      }
      if (erow == 0)
        ok_s[it & 1] = mbar_wait(tfull, aphase, p.status, wait_limit(p)) &&
                               !(p.test_timeout && !mbar_wait(never, 0, p.status, wait_limit(p)))
                           ? 1
                           : 0;
      if (WFMT == 0) {
        const int n = head * 128 + row;
        ws_s[((it & 1) * 2 + wg) * 128 + row] = n < p.N ? __ldg(p.w_scale + n) : 0.f;
      }
      named_bar_sync(1, kEpiThreads);
      if (!ok_s[it & 1]) break;
      tc_fence_after();
      float v[128];
      const uint32_t base = tmem + ((uint32_t)((warp & 3) * 32) << 16) + wg * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float part[32];
        tc_ld32(base + c * 32, part);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[c * 32 + i] = part[i];
      }
      tc_wait_ld();
      tc_fence_before();
      // the warpgroup's accumulator columns are in registers: one arrival
      // tells CTA 0's MMA issuer it may overwrite them (one remote arrival per
      // thread would serialise hundreds of them on one barrier).  Relaxed:
      // the reads it releases have completed (tcgen05.wait::ld, then the
      // warpgroup barrier), and a release would first wait for the previous
      // tile's output stores (measured: the issuer waited ~1.2 us a tile)
      named_bar_sync(2 + wg, 128);
      if ((warp & 3) == 0 && lane == 0) arrive_remote_relaxed(tempty0);
      aphase ^= 1;
      if (WFMT == 0 && live) {
        const float *wsb = ws_s + ((it & 1) * 2 + wg) * 128;
#pragma unroll
        for (int i = 0; i < 128; ++i) v[i] = v[i] * xs * wsb[i];
      }
      HeadCtx hc;
      hc.m = m;
      hc.head = head;
      hc.cs_row = p.cos_sin + pos * kRotDim;
      hc.slot = slot;
      hc.islot = islot;
      hc.g_q = p.g_q;
      hc.g_k = p.g_k;
      hc.g_iq = p.g_iq;
      hc.g_ik = p.g_ik;
      if (p.cache_fmt == 0 && head >= p.v0 && head < p.iq0) {  // the warpgroup's head is a V head
        v_rows_fp8_warp(p, hc, v, live);                       // every lane of the warp
        continue;
      }
      if (!live) continue;
      head_epilogue<128>(p, hc, v, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair may still signal it
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

}  // namespace g2

// ------------------------------------------------------------------- host

cudaError_t launch_gemm_pair(const Params &p, int num_sms, int64_t l2_bytes, int grid_override, bool pdl,
                             cudaStream_t stream) {
  if (p.H % g2::kBK || p.N % 128) return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB, tmSFA, tmSFB;
  const int ksf = p.H / 32;
  if (!map_rows_sw128(&tmA, p.xq, p.M, p.H, g2::kBK, 128) || !map_rows_sw128(&tmB, p.w, p.N, p.H, g2::kBK, 128))
    return cudaErrorInvalidValue;
  if (p.weight_fmt == 1) {
    if (!map_scale_atoms(&tmSFA, p.xsf, p.m_pad / 128, ksf) || !map_scale_atoms(&tmSFB, p.wsf, p.N / 128, ksf))
      return cudaErrorInvalidValue;
  } else {
    tmSFA = tmA;  // unused by the per-channel kernel
    tmSFB = tmB;
  }
  g2::Sched sc;
  sc.m_pairs = (p.M + 255) / 256;
  sc.n_tiles = (p.N + g2::kBN - 1) / g2::kBN;
  sc.ksteps = p.H / g2::kBK;
  const int tiles = sc.m_pairs * sc.n_tiles;
  int clusters = (grid_override > 0 ? grid_override : num_sms) / 2;
  if (clusters < 1) clusters = 1;
  if (clusters > tiles) clusters = tiles;
  // raster groups: a group's activation rows (256 a pair, K bytes each) take
  // at most a quarter of the L2
  const int64_t per_pair = (int64_t)256 * p.H;
  const int64_t gm = (l2_bytes / 4) / (per_pair > 0 ? per_pair : 1);
  sc.group_m = gm < 1 ? 1 : (gm > sc.m_pairs ? sc.m_pairs : (int)gm);
  auto kern = p.weight_fmt == 0 ? g2::pa_gemm_pair_kernel<0> : g2::pa_gemm_pair_kernel<1>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), g2::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(g2::kThreads);
  cfg.dynamicSmemBytes = g2::kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmSFA, tmSFB, p, sc, (int)pdl);
}

}  // namespace pa
