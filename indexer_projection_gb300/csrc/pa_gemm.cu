// Tensor-core path of the pre-attention projection (M > 16): a persistent,
// warp-specialised tcgen05 GEMM with the per-head epilogue fused behind the
// TMEM accumulator, so the [M, N] projection never reaches memory.
//
//   tile      BM x BN x BK = 128 x 128 x 128: one M-tile of token rows by one
//             128-column head ("vllm.models.minimax_m3.nvidia.ops.
//             qkv_index_fused_epilogue", QkvIndexFusedEpilogueKernel: one
//             head per epilogue warpgroup)
//   warp 0-3  epilogue: thread i owns tile row i (TMEM lane i); drains its
//             128 f32 columns with tcgen05.ld, then Gemma RMSNorm, RoPE,
//             quantisation and the paged scatter in registers
//   warp 4    TMA producer: A (activations) and B (weights) 128x128-byte
//             tiles, 128B-swizzled, into an S-stage ring; for MXFP8 also the
//             512-byte F8_128x4 scale atoms of both operands (1-D bulk copies)
//   warp 5    TMEM allocator and MMA issuer: per k-step 4 x
//             tcgen05.mma m128 n128 k32 (kind::f8f6f4, or
//             kind::mxf8f6f4.block_scale with the scale atoms moved to TMEM by
//             tcgen05.cp and the K-block picked by the instruction's SF id)
//   TMEM      two 128-column accumulators (the epilogue of tile i overlaps the
//             MMAs of tile i + 1) and 8 scale-factor columns
//
// The per-channel format applies x_scale[m] * w_scale[n] in the epilogue
// ("vllm.models.minimax_m3.amd.mono.kernels.pre_attn", GEMV tasks); MXFP8
// applies 2^(e_a + e_b) per 32-block inside the MMA.
//
// Every mbarrier wait is bounded (about a second); a timeout raises
// PA_DEV_WAIT_TIMEOUT, and the kernel still finishes and frees its TMEM.
#include "pa_device.cuh"
#include "pa_launch.h"
#include "pa_tc.cuh"
#include "pa_tma.h"

namespace pa {

constexpr int kBM = 128, kBN = 128, kBK = 128;
constexpr int kStages = 6;
constexpr int kTileBytes = kBM * kBK;  // 16 KB per operand tile (e4m3)
constexpr int kSfBytes = 512;          // one F8_128x4 atom: 128 rows x 4 K-blocks
constexpr int kGemmThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kSfaCol = 256, kSfbCol = 260;
// Instruction descriptors (M = 128, N = 128, A and B E4M3, K-major).
constexpr uint32_t kIdescF8 = idesc_f8(kBM, kBN);
constexpr uint32_t kIdescMx = idesc_mx(kBM, kBN);

struct GemmSmem {  // offsets from the 1024-aligned base
  static constexpr int a = 0;
  static constexpr int b = a + kStages * kTileBytes;
  static constexpr int sfa = b + kStages * kTileBytes;
  static constexpr int sfb = sfa + kStages * kSfBytes;
  static constexpr int bars = sfb + kStages * kSfBytes;  // full[S], empty[S], tfull[2], tempty[2], never, drain
  static constexpr int tmem_addr = bars + (2 * kStages + 6) * 8;
  static constexpr int ok = tmem_addr + 8;                // 2 x int: tile verdicts
  static constexpr int wscale = ok + 8;                   // 2 x 128 f32: per-channel weight scales of a head
  static constexpr int total = wscale + 2 * kBN * 4;
};
constexpr int kGemmSmemBytes = GemmSmem::total + 1024;  // + alignment slack

// 2-D TMA tile load (x = K byte offset, y = row) completing on `bar`.
__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

template <int WFMT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    pa_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, Params p,
                int use_pdl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + GemmSmem::bars);
  uint64_t *empty = full + kStages;
  uint64_t *tfull = empty + kStages;
  uint64_t *tempty = tfull + 2;
  uint64_t *never = tempty + 2;  // testing: nothing arrives on it
  uint64_t *drain = never + 1;   // the MMA issuer's last commit on an abnormal exit
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + GemmSmem::tmem_addr);
  float *ws_s = reinterpret_cast<float *>(smem + GemmSmem::wscale);
  volatile int *ok_s = reinterpret_cast<volatile int *>(smem + GemmSmem::ok);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = p.M, K = p.H;
  const int m_tiles = (M + kBM - 1) / kBM, n_tiles = p.N / kBN;
  const int tiles = m_tiles * n_tiles;
  const int ksteps = K / kBK;
  const int ksf = K >> 5;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kBM / 32);  // one arrival per epilogue warp
    }
    mbar_init(never, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (use_pdl) {
    pdl_trigger();
    pdl_wait();
  }

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t tx = 2 * kTileBytes + (WFMT == 1 ? 2 * kSfBytes : 0);
      bool ok = true;
      int last_ph[kStages];  // phase each stage was last loaded with (-1: never)
#pragma unroll
      for (int i = 0; i < kStages; ++i) last_ph[i] = -1;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int mt = t / n_tiles, nt = t - mt * n_tiles;
        for (int ks = 0; ks < ksteps; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.status, wait_limit(p))) {
            ok = false;
            break;
          }
          last_ph[stage] = (int)phase;
          mbar_expect_tx(&full[stage], tx);
          tma_2d(smem + GemmSmem::a + stage * kTileBytes, &tmA, ks * kBK, mt * kBM, &full[stage]);
          tma_2d(smem + GemmSmem::b + stage * kTileBytes, &tmB, ks * kBK, nt * kBN, &full[stage]);
          if (WFMT == 1) {
            bulk_g2s(smem + GemmSmem::sfa + stage * kSfBytes, p.xsf + ((int64_t)mt * (ksf >> 2) + ks) * kSfBytes,
                     kSfBytes, &full[stage]);
            bulk_g2s(smem + GemmSmem::sfb + stage * kSfBytes, p.wsf + ((int64_t)nt * (ksf >> 2) + ks) * kSfBytes,
                     kSfBytes, &full[stage]);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // a wait ran out: the copies already issued land before the CTA exits
      if (!ok)
#pragma unroll
        for (int i = 0; i < kStages; ++i)
          if (last_ph[i] >= 0) mbar_wait(&full[i], (uint32_t)last_ph[i], p.status, wait_limit(p));
    }
  } else if (warp == 5) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int abuf = 0;
      uint32_t aphase = 0;
      bool ok = true;
      const uint32_t a0 = smem_u32(smem + GemmSmem::a), b0 = smem_u32(smem + GemmSmem::b);
      const uint32_t sfa0 = smem_u32(smem + GemmSmem::sfa), sfb0 = smem_u32(smem + GemmSmem::sfb);
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        if (!mbar_wait(&tempty[abuf], aphase ^ 1, p.status, wait_limit(p))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dacc = tmem + abuf * kBN;
        for (int ks = 0; ks < ksteps; ++ks) {
          if (!mbar_wait(&full[stage], phase, p.status, wait_limit(p))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(a0 + stage * kTileBytes), bd = sdesc_sw128(b0 + stage * kTileBytes);
          if (WFMT == 1) {
            tc_cp_sf(tmem + kSfaCol, sdesc_sf(sfa0 + stage * kSfBytes));
            tc_cp_sf(tmem + kSfbCol, sdesc_sf(sfb0 + stage * kSfBytes));
          }
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k) {
            const uint32_t acc = (ks | k) != 0;
            // +32 bytes along K inside the 128-byte swizzle atom: +2 in the
            // descriptor's 16-byte address field
            if (WFMT == 0) {
              mma_f8(dacc, ad + 2 * k, bd + 2 * k, kIdescF8, acc);
            } else {
              const uint32_t idesc = kIdescMx | ((uint32_t)k << 4) | ((uint32_t)k << 29);
              mma_mx(dacc, ad + 2 * k, bd + 2 * k, idesc, tmem + kSfaCol, tmem + kSfbCol, acc);
            }
          }
          tc_commit(&empty[stage]);  // the stage is free once these MMAs have read it
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        tc_commit(&tfull[abuf]);
        if (++abuf == 2) {
          abuf = 0;
          aphase ^= 1;
        }
      }
      if (!ok) {  // a wait ran out: the MMAs already issued complete before the TMEM is freed
        tc_commit(drain);
        mbar_wait(drain, 0, p.status, wait_limit(p));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int row = threadIdx.x;  // 0..127: TMEM lane and tile row
    int abuf = 0;
    uint32_t aphase = 0;
    int it = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
      const int mt = t / n_tiles, nt = t - mt * n_tiles;
      // the row's position, slots and scale, and its cos / sin line, fetched
      // while the tile's MMAs run (they do not depend on them)
      const int m = mt * kBM + row;
      const bool live = m < M;
      int64_t pos = 0, slot = -1, islot = -1;
      float xs = 1.0f;
      if (live) {
        pos = load_pos(p, m);
        slot = ld_i64(p.slot + m);
        islot = ld_i64(p.islot + m);
        if (WFMT == 0) xs = __ldcg(p.x_scale + m);
        asm volatile("prefetch.global.L1 [%0];" ::"l"(p.cos_sin + pos * kRotDim));
      }
      // one thread waits; the verdict and the head's per-channel weight
      // scales are shared through double-buffered shared memory
      if (row == 0)
        ok_s[it & 1] = mbar_wait(&tfull[abuf], aphase, p.status, wait_limit(p)) &&
                               !(p.test_timeout && !mbar_wait(never, 0, p.status, wait_limit(p)))
                           ? 1
                           : 0;
      if (WFMT == 0) ws_s[(it & 1) * kBN + row] = __ldg(p.w_scale + nt * kBN + row);
      named_bar(1, kBM);
      if (!ok_s[it & 1]) break;
      tc_fence_after();
      float v[kBN];
      const uint32_t base = tmem + ((uint32_t)(warp * 32) << 16) + abuf * kBN;
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        float part[32];
        tc_ld32(base + c * 32, part);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[c * 32 + i] = part[i];
      }
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[abuf]);
      if (++abuf == 2) {
        abuf = 0;
        aphase ^= 1;
      }
      if (WFMT == 0 && live) {
        const float *wsb = ws_s + (it & 1) * kBN;
#pragma unroll
        for (int i = 0; i < kBN; ++i) v[i] = v[i] * xs * wsb[i];
      }
      HeadCtx hc;
      hc.m = m;
      hc.head = nt;
      hc.cs_row = p.cos_sin + pos * kRotDim;
      hc.slot = slot;
      hc.islot = islot;
      hc.g_q = p.g_q;
      hc.g_k = p.g_k;
      hc.g_iq = p.g_iq;
      hc.g_ik = p.g_ik;
      if (p.cache_fmt == 0 && nt >= p.v0 && nt < p.iq0) {  // a V head
        v_rows_fp8_warp(p, hc, v, live);                   // every lane of the warp
        continue;
      }
      if (!live) continue;
      head_epilogue<kBN>(p, hc, v, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ------------------------------------------------------------------- host

cudaError_t launch_gemm(const Params &p, int num_sms, int grid_override, bool pdl, cudaStream_t stream) {
  if (p.H % kBK || p.N % kBN) return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB;
  if (!map_rows_sw128(&tmA, p.xq, p.M, p.H, kBK, kBM) || !map_rows_sw128(&tmB, p.w, p.N, p.H, kBK, kBN))
    return cudaErrorInvalidValue;
  const int tiles = ((p.M + kBM - 1) / kBM) * (p.N / kBN);
  int grid = grid_override > 0 ? grid_override : num_sms;
  if (grid > tiles) grid = tiles;
  auto kern = p.weight_fmt == 0 ? pa_gemm_kernel<0> : pa_gemm_kernel<1>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), kGemmSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = kGemmSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p, (int)pdl);
}

}  // namespace pa
