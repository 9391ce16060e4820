// Device-side building blocks of the pre-attention step for sm_103a:
// kernel parameters, PTX wrappers (mbarrier, bulk copies, programmatic
// dependent launch, thread-block clusters), FP8 / FP4 codecs
// and the per-head epilogue (Gemma RMSNorm, partial NeoX RoPE, q / index_q
// outputs, FP8 and NVFP4 paged-cache insertion).
//
// Pages cited:
//   [K1]  "vllm.models.minimax_m3.amd.mono.kernels.pre_attn" (K1 mono_pre)
//   [EPI] "vllm.models.minimax_m3.nvidia.ops.qkv_index_fused_epilogue"
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

constexpr int kHeadDim = 128;
constexpr int kRotDim = 64;
constexpr int kHalfRot = 32;
constexpr float kFp8Max = 448.0f;
constexpr uint32_t kDevSlotRange = 1u << 0;
constexpr uint32_t kDevPosRange = 1u << 1;
constexpr uint32_t kDevWaitTimeout = 1u << 2;

// Everything a kernel of the step reads or writes.  Passed by value.
struct Params {
  int M, H, N, n_heads;
  int n_q, n_kv, n_iq;
  int k0, v0, iq0, ik0;  // first head of each role
  int weight_fmt;        // 0 per-channel FP8, 1 MXFP8
  int cache_fmt;         // 0 FP8, 1 NVFP4
  int bs;                // tokens per page
  int kps;               // FP8 page16_of stride (8 = identity)
  int static_kv;         // FP8 caches: K / V scale fixed at 1
  int exact_norm;        // testing: the prologue's exact path for every element
  float eps;
  // inputs
  const __nv_bfloat16 *ar, *res, *g_in;
  const uint8_t *w;
  const float *w_scale;      // per-channel [N]
  const uint8_t *wsf;        // MXFP8, F8_128x4 layout of [N, H/32]
  const __nv_bfloat16 *g_q, *g_k, *g_iq, *g_ik, *cos_sin;
  int64_t max_pos;
  const int64_t *pos, *slot, *islot;
  // caches
  uint8_t *k_cache, *v_cache, *index_cache;
  float *k_scale, *v_scale;
  int64_t num_pages16, num_index_slots;
  uint8_t *kv_cache, *idx_cache;
  int64_t kv_pages, kv_page_bytes, idx_pages, idx_page_bytes;
  float k_gs_inv, v_gs_inv;  // 1 / global NVFP4 scales (f32 reciprocal)
  // outputs
  __nv_bfloat16 *residual, *q, *iq;
  uint8_t *q_fp8, *iq_fp8;
  float q_fp8_inv;           // 1 / q_fp8_scale (f32 reciprocal)
  uint32_t *done;            // [M, n_heads] done words (NULL: none), set to done_epoch
  uint32_t done_epoch;
  int test_timeout;          // testing: a wait that cannot complete, with a short limit
  // workspace
  uint32_t *status;
  uint8_t *xq;               // [M, H] e4m3 activations
  float *x_scale;            // [M] per-token scales (per-channel format)
  uint8_t *xsf;              // MXFP8 activation scales, F8_128x4 of [Mpad, H/32]
  int m_pad;                 // M rounded up to 128 (MXFP8 scale rows)
};

// ------------------------------------------------------------ small utils

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
// f32 -> bf16 bits (round to nearest even), one value a conversion.
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
// Two f32 -> two bf16 (round to nearest even), lo in the low half, in one
// packed conversion (on sm_103a it converts about four times as many values
// a cycle as the single-value conversion).
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// bf16_round of a pair, through one packed conversion.
__device__ __forceinline__ void bf16_round2(float a, float b, float &ra, float &rb) {
  const uint32_t w = bf16x2_bits(a, b);
  ra = __uint_as_float(w << 16);
  rb = __uint_as_float(w & 0xffff0000u);
}

// Two f32 -> two E4M3 (round to nearest even, saturate to +-448); lo in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return (uint32_t)e4m3x2(a, b) | ((uint32_t)e4m3x2(c, d) << 16);
}
__device__ __forceinline__ uint8_t e4m3(float a) { return (uint8_t)(e4m3x2(a, 0.0f) & 0xff); }
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)c));
  return __half2float(__ushort_as_half((uint16_t)(h & 0xffff)));
}
// Two f32 -> two E2M1 nibbles (round to nearest even, saturate to +-6); lo in bits 0-3.
__device__ __forceinline__ uint8_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{.reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t;}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return (uint8_t)r;
}
// f32 product rounded toward zero ([EPI] _nvfp4_quant32).
__device__ __forceinline__ float mul_rz(float a, float b) { return __fmul_rz(a, b); }

__device__ __forceinline__ void set_status(uint32_t *st, uint32_t bit) { atomicOr(st, bit); }
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ int64_t ld_i64(const int64_t *p) { return __ldg(p); }
// A hint that brings the line into L2 (and its translation into the TLBs).
// It orders nothing and changes no value a later load returns, so it may be
// issued for an input before the wait on the kernel that produces it.
__device__ __forceinline__ void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// Offset of (row r, K-block kb) in the F8_128x4 scale layout ([EPI]
// prepare_SF): [R/128, Ksf/4, 32, 4, 4].
__device__ __forceinline__ int64_t sf128x4_offset(int64_t r, int kb, int ksf) {
  return ((r >> 7) * (ksf >> 2) + (kb >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (kb & 3);
}

// ------------------------------------------------ programmatic dependent launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p;}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Limit of every bounded device wait: about a second; with the testing flag
// PA_FLAG_TEST_WAIT_TIMEOUT, kTestWaitNs (every wait of the kernels is then
// short enough for a test to run one out on purpose).
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint64_t kTestWaitNs = 200000ull;
__device__ __forceinline__ uint64_t wait_limit(const Params &p) { return p.test_timeout ? kTestWaitNs : kWaitNs; }

// Wait for phase `parity` of an mbarrier, giving up after limit_ns: the
// caller's results are then invalid and PA_DEV_WAIT_TIMEOUT is raised.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *status,
                                          uint64_t limit_ns = kWaitNs) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (globaltimer() - t0 > limit_ns) {
      set_status(status, kDevWaitTimeout);
      return false;
    }
  }
}

// ------------------------------------------- asynchronous global -> shared
// (cp.async: no registers held while the copy is in flight; .cg bypasses L1,
// so data written by the previous kernel is read from L2)
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------ thread-block clusters
__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// This CTA's shared address `saddr` as seen in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Arrive on an mbarrier given by its cluster address, without release
// semantics: for an arrival that orders nothing in memory the waiter reads
// (a tensor-memory accumulator freed after tcgen05.wait::ld and
// tcgen05.fence::before_thread_sync).  A release there would wait until every
// earlier store of the thread is performed at cluster scope, which behind an
// epilogue's global stores takes microseconds.
__device__ __forceinline__ void arrive_remote_relaxed(uint32_t caddr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
// Asynchronous store of 16 bytes into the shared memory of a CTA of the
// cluster; its completion counts 16 bytes on that CTA's mbarrier `cbar`
// (both addresses in the destination CTA, as given by mapa).
__device__ __forceinline__ void st_async_v4(uint32_t caddr, float4 v, uint32_t cbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1,%2,%3,%4}, [%5];" ::"r"(caddr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(cbar)
               : "memory");
}
// Wait for phase `parity` of a local mbarrier whose arrivals come from other
// CTAs of the cluster (acquire at cluster scope), giving up after limit_ns
// (PA_DEV_WAIT_TIMEOUT).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, uint32_t *status,
                                                  uint64_t limit_ns = kWaitNs) {
  const uint32_t a = smem_u32(bar);
  auto try_wait = [&]() {
    uint32_t ok;
    asm volatile(
        "{.reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p;}"
        : "=r"(ok) : "r"(a), "r"(parity) : "memory");
    return ok != 0;
  };
  if (try_wait()) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (try_wait()) return true;
    if (globaltimer() - t0 > limit_ns) {
      set_status(status, kDevWaitTimeout);
      return false;
    }
  }
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ================================================================ epilogue
//
// One 128-dim head row of one token is held by G = 128 / E consecutive lanes,
// E consecutive dims each (E = 4: a warp per row, as the pre_attn page's half
// wave; E = 128: a thread per row, as the epilogue page's TMEM drain).
template <int E>
struct Row {
  static constexpr int G = kHeadDim / E;
  static_assert(G >= 1 && G <= 32 && (G & (G - 1)) == 0, "E must divide 128");
  __device__ static __forceinline__ float sum(float x) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
  }
  __device__ static __forceinline__ float max(float x) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
  }
};

// Gemma RMSNorm of a head row in place: v * rsqrt(mean(v^2) + eps) * (1 + gamma)
// ([K1] head_norm_rope, [EPI] _rms_norm).
template <int E>
__device__ __forceinline__ void head_rmsnorm(float (&v)[E], int d0, const __nv_bfloat16 *gamma, float eps) {
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) ss = fmaf(v[i], v[i], ss);
  ss = Row<E>::sum(ss);
  const float rr = rsqrtf(ss * (1.0f / kHeadDim) + eps);
  const uint2 *g = reinterpret_cast<const uint2 *>(gamma + d0);
#pragma unroll
  for (int q = 0; q < E / 4; ++q) {
    const uint2 gw = g[q];
    float gg[4] = {bf16_to_f32(gw.x & 0xffff), bf16_to_f32(gw.x >> 16), bf16_to_f32(gw.y & 0xffff),
                   bf16_to_f32(gw.y >> 16)};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float n = v[4 * q + j] * rr;
      v[4 * q + j] = fmaf(n, gg[j], n);
    }
  }
}

// Partial NeoX RoPE over dims [0, 64) ([K1] head_norm_rope, [EPI] _rope64):
// x' = x c - y s, y' = y c + x s with x = dim i, y = dim i + 32, c / s the
// bf16 cos_sin[pos][i], cos_sin[pos][32 + i].
template <int E>
__device__ __forceinline__ void head_rope(float (&v)[E], int d0, const __nv_bfloat16 *cs_row) {
  if constexpr (E >= kRotDim) {
    // the thread holds dims [d0, d0 + E); d0 = 0 whenever it holds [0, 64)
    if (d0 == 0) {
      // 16-byte pieces of the (16-byte aligned) cos / sin row: with a thread
      // a row, every load instruction touches as many lines as the warp has
      // rows, so fewer and wider loads
      const uint4 *cs4 = reinterpret_cast<const uint4 *>(cs_row);
#pragma unroll
      for (int q = 0; q < kHalfRot / 8; ++q) {
        const uint4 cq = cs4[q], sq = cs4[kHalfRot / 8 + q];
        const uint32_t cw4[4] = {cq.x, cq.y, cq.z, cq.w}, sw4[4] = {sq.x, sq.y, sq.z, sq.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = 8 * q + 2 * k;
          const uint32_t cw = cw4[k], sw = sw4[k];
          float c[2] = {bf16_to_f32(cw & 0xffff), bf16_to_f32(cw >> 16)};
          float s[2] = {bf16_to_f32(sw & 0xffff), bf16_to_f32(sw >> 16)};
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float x = v[i + j], y = v[i + j + kHalfRot];
            v[i + j] = x * c[j] - y * s[j];
            v[i + j + kHalfRot] = y * c[j] + x * s[j];
          }
        }
      }
    }
  } else {
    // partner dims (i +- 32) sit 32 / E lanes away
    constexpr int kLanes = kHalfRot / E;
    const bool first = d0 < kHalfRot;
    const bool in_rope = d0 < kRotDim;
    const int ib = first ? d0 : d0 - kHalfRot;
    float c[E], s[E];
    if (in_rope) {
#pragma unroll
      for (int j = 0; j < E; ++j) {
        c[j] = __bfloat162float(cs_row[ib + j]);
        s[j] = __bfloat162float(cs_row[kHalfRot + ib + j]);
      }
    }
#pragma unroll
    for (int j = 0; j < E; ++j) {
      float p = __shfl_xor_sync(0xffffffffu, v[j], kLanes);
      if (in_rope) v[j] = first ? (v[j] * c[j] - p * s[j]) : (v[j] * c[j] + p * s[j]);
    }
  }
}

// e4m3 codes of RN(x / s) (s > 0) for 4 values, from the product with
// rs = RN(1 / s): x * rs is within 2^-22 (relative) of x / s and of its
// rounding, so where the codes of x * rs scaled by 1 -+ 2^-20 agree, every
// value in between (RN(x / s) included) has that code, rounding being
// monotonic.  `ok` is cleared otherwise (a value within 2^-20 of a code
// boundary, about one in 2^15), and the caller then takes the true quotient
// (e4m3x4_div): the codes are those of the division bit for bit.  The check
// and the rare division are kept apart so the common path stays straight-line
// code (a fused select of the two measured 6x slower in a thread-per-row
// epilogue).
__device__ __forceinline__ uint32_t e4m3x4_prod_checked(float a, float b, float c, float d, float rs, bool &ok) {
  const float qa = a * rs, qb = b * rs, qc = c * rs, qd = d * rs;
  constexpr float lo = 1.0f - 0x1p-20f, hi = 1.0f + 0x1p-20f;
  const uint32_t w = e4m3x4(qa, qb, qc, qd);
  const uint32_t wl = e4m3x4(qa * lo, qb * lo, qc * lo, qd * lo), wh = e4m3x4(qa * hi, qb * hi, qc * hi, qd * hi);
  ok = ok & (w == wl) & (w == wh);
  return w;
}
static __device__ __noinline__ uint32_t e4m3x4_div(float a, float b, float c, float d, float s) {
  return e4m3x4(__fdiv_rn(a, s), __fdiv_rn(b, s), __fdiv_rn(c, s), __fdiv_rn(d, s));
}

// [K1] page16_of: page-16 id of a slot under the K / V block page stride.
__device__ __forceinline__ int64_t page16_of(int64_t slot, int kps) {
  if (kps == 8) return slot >> 4;
  return (slot >> 7) * kps + ((slot & 127) >> 4);
}

// NVFP4 group quantiser ([EPI] _nvfp4_quant32) for 4 values of a 16-dim
// group whose max magnitude is gmax: returns the scale byte, fills two
// packed bytes (even dim in the low nibble, zero magnitudes unsigned).
__device__ __forceinline__ uint8_t nvfp4_scale(float gmax, bool has_gs, float gs_inv, float &r) {
  float a = gmax * (1.0f / 6.0f);
  if (has_gs) a = a * gs_inv;
  a = fmaxf(a, 0x1p-9f);
  const uint8_t sf = e4m3(a);
  r = __frcp_rn(e4m3_to_f32(sf));
  if (has_gs) r = r * gs_inv;
  return sf;
}
__device__ __forceinline__ uint16_t nvfp4_quad(const float *v4, float r) {
  uint32_t b0 = e2m1x2(mul_rz(v4[0], r), mul_rz(v4[1], r));
  uint32_t b1 = e2m1x2(mul_rz(v4[2], r), mul_rz(v4[3], r));
  uint32_t w = b0 | (b1 << 8);
  const uint32_t m = 0x7777u;
  w = w & (((w & m) + m) | m);  // clear the sign of zero magnitudes
  return (uint16_t)w;
}

// Everything the epilogue of one (token, head) needs besides the values.
// The gamma and cos/sin pointers may point to global or shared memory.
struct HeadCtx {
  int m;        // token row
  int head;     // head index in [0, n_heads)
  int64_t slot, islot;
  const __nv_bfloat16 *cs_row;            // cos_sin row of the token's (clamped) position
  const __nv_bfloat16 *g_q, *g_k, *g_iq, *g_ik;
};

__device__ __forceinline__ int64_t load_pos(const Params &p, int m) {
  int64_t pos = ld_i64(p.pos + m);
  if (pos < 0 || pos >= p.max_pos) {
    set_status(p.status, kDevPosRange);
    pos = pos < 0 ? 0 : p.max_pos - 1;
  }
  return pos;
}

// Run the role logic of one head row.  v: this thread's E values (dims
// d0 .. d0 + E - 1) of the f32 projection.  Heads are
// [q x n_q | k x n_kv | v x n_kv | index_q x n_iq | index_k]
// ([EPI] QkvIndexFusedEpilogueKernel.__init__); per role ([K1] head tasks,
// [EPI] kernel epilogue):
//   q       norm + rope -> bf16 and / or e4m3(z * (1/q_fp8_scale))
//   k       norm + rope -> FP8: e4m3(bf16(z) / ks), ks = amax / 448;
//                          NVFP4 with 1/k_global, linear scale bytes
//   v       raw         -> FP8: e4m3(y / vs);  NVFP4 with 1/v_global, V-swizzled scales
//   index_q norm + rope -> bf16 and / or e4m3(z)
//   index_k norm + rope -> FP8: e4m3(bf16(z)) in the index cache; NVFP4 unit scale
// A slot < 0 skips that cache; a slot beyond the cache skips it and flags.
// CF: the cache format when known at compile time (0 FP8, 1 NVFP4; the other
// format's code is then left out of the kernel), else -1 (p.cache_fmt).
template <int E, int CF = -1>
__device__ __forceinline__ void head_epilogue_stores(const Params &p, const HeadCtx &hc, float (&v)[E], int d0) {
  const int h = hc.head;
  const bool is_q = h < p.k0, is_k = h >= p.k0 && h < p.v0, is_v = h >= p.v0 && h < p.iq0;
  const bool is_iq = h >= p.iq0 && h < p.ik0;
  if (!is_v) {
    const __nv_bfloat16 *g = is_q ? hc.g_q : is_k ? hc.g_k : is_iq ? hc.g_iq : hc.g_ik;
    head_rmsnorm<E>(v, d0, g, p.eps);
    head_rope<E>(v, d0, hc.cs_row);
  }
  const int m = hc.m;
  if (is_q || is_iq) {
    const int nh = is_q ? p.n_q : p.n_iq;
    const int j = is_q ? h : h - p.iq0;
    __nv_bfloat16 *ob = is_q ? p.q : p.iq;
    uint8_t *of = is_q ? p.q_fp8 : p.iq_fp8;
    const float sc = is_q ? p.q_fp8_inv : 1.0f;
    const int64_t base = (int64_t)m * nh * kHeadDim + (int64_t)j * kHeadDim + d0;
    // a thread holding a whole row (E >= 16) stores 16 bytes at a time (a
    // quarter of the store transactions of 4-byte pieces); a warp holding a
    // row (E = 4) already writes it contiguously
    if (ob) {
      // A thread holding a whole row (the tensor-core epilogues, which run
      // beside the next tile's K loop) converts one value at a time: with the
      // packed conversion that epilogue was faster but the prefill GEMM 4%
      // slower (measured on the same GPU; the cause was not pinned down)
      auto bf2 = [&](int i) {
        if constexpr (E >= 8)
          return (uint32_t)f32_to_bf16_bits(v[i]) | ((uint32_t)f32_to_bf16_bits(v[i + 1]) << 16);
        else
          return bf16x2_bits(v[i], v[i + 1]);
      };
      if constexpr (E >= 8) {
#pragma unroll
        for (int q = 0; q < E / 8; ++q)
          *reinterpret_cast<uint4 *>(ob + base + 8 * q) =
              make_uint4(bf2(8 * q), bf2(8 * q + 2), bf2(8 * q + 4), bf2(8 * q + 6));
      } else {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) *reinterpret_cast<uint2 *>(ob + base + 4 * q) = make_uint2(bf2(4 * q), bf2(4 * q + 2));
      }
    }
    if (of) {
      auto f8x4 = [&](int i) {
        return is_q ? e4m3x4(v[i] * sc, v[i + 1] * sc, v[i + 2] * sc, v[i + 3] * sc)
                    : e4m3x4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      };
      if constexpr (E >= 16) {
#pragma unroll
        for (int q = 0; q < E / 16; ++q)
          *reinterpret_cast<uint4 *>(of + base + 16 * q) =
              make_uint4(f8x4(16 * q), f8x4(16 * q + 4), f8x4(16 * q + 8), f8x4(16 * q + 12));
      } else {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) *reinterpret_cast<uint32_t *>(of + base + 4 * q) = f8x4(4 * q);
      }
    }
    return;
  }
  const bool is_ik = !is_k && !is_v;
  const int64_t slot = is_ik ? hc.islot : hc.slot;
  if (slot < 0) return;
  if ((CF >= 0 ? CF : p.cache_fmt) == 0) {
    // ---------------------------------------------------------- FP8 caches
    if (is_ik) {
      if (slot >= p.num_index_slots) {
        if (d0 == 0) set_status(p.status, kDevSlotRange);
        return;
      }
      uint8_t *dst = p.index_cache + slot * kHeadDim + d0;
      auto ik4 = [&](int i) {
        float a, b, c, d;
        bf16_round2(v[i], v[i + 1], a, b);
        bf16_round2(v[i + 2], v[i + 3], c, d);
        return e4m3x4(a, b, c, d);
      };
      if constexpr (E >= 16) {
#pragma unroll
        for (int q = 0; q < E / 16; ++q)
          *reinterpret_cast<uint4 *>(dst + 16 * q) = make_uint4(ik4(16 * q), ik4(16 * q + 4), ik4(16 * q + 8), ik4(16 * q + 12));
      } else {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) *reinterpret_cast<uint32_t *>(dst + 4 * q) = ik4(4 * q);
      }
      return;
    }
    const int kvh = is_k ? h - p.k0 : h - p.v0;
    const int64_t p16 = page16_of(slot, p.kps);
    if (p16 >= p.num_pages16) {
      if (d0 == 0) set_status(p.status, kDevSlotRange);
      return;
    }
    const int t = (int)(slot & 15);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = Row<E>::max(amax);
    const float s = p.static_kv ? 1.0f : (amax == 0.f ? 1.0f : __fdiv_rn(amax, kFp8Max));
    const float rs = __frcp_rn(s);
    const int64_t page = (p16 * p.n_kv + kvh) * 2048;
    if (is_k) {
      // codes of 4 K values (bf16 first), the true quotient only where the
      // product's code is not certain
      auto k4 = [&](int i, bool &ok) {
        float a, b, c, d;
        bf16_round2(v[i], v[i + 1], a, b);
        bf16_round2(v[i + 2], v[i + 3], c, d);
        return e4m3x4_prod_checked(a, b, c, d, rs, ok);
      };
      auto k4_div = [&](int i) {
        float a, b, c, d;
        bf16_round2(v[i], v[i + 1], a, b);
        bf16_round2(v[i + 2], v[i + 3], c, d);
        return e4m3x4_div(a, b, c, d, s);
      };
      if constexpr (E >= 16) {  // 16 dims: one 16-byte row of the page's 16 x 16 block
#pragma unroll
        for (int q = 0; q < E / 16; ++q) {
          const int d = d0 + 16 * q;
          bool ok = true;
          uint4 w = make_uint4(k4(16 * q, ok), k4(16 * q + 4, ok), k4(16 * q + 8, ok), k4(16 * q + 12, ok));
          if (__builtin_expect(!ok, 0))
            w = make_uint4(k4_div(16 * q), k4_div(16 * q + 4), k4_div(16 * q + 8), k4_div(16 * q + 12));
          *reinterpret_cast<uint4 *>(p.k_cache + page + (d >> 4) * 256 + t * 16) = w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) {
          const int d = d0 + 4 * q;
          bool ok = true;
          uint32_t w = k4(4 * q, ok);
          if (__builtin_expect(!ok, 0)) w = k4_div(4 * q);
          *reinterpret_cast<uint32_t *>(p.k_cache + page + (d >> 4) * 256 + t * 16 + (d & 15)) = w;
        }
      }
      if (d0 == 0) p.k_scale[(p16 * p.n_kv + kvh) * 16 + t] = s;
    } else {
#pragma unroll
      for (int i = 0; i < E; i += 4) {
        bool ok = true;
        uint32_t w = e4m3x4_prod_checked(v[i], v[i + 1], v[i + 2], v[i + 3], rs, ok);
        if (__builtin_expect(!ok, 0)) w = e4m3x4_div(v[i], v[i + 1], v[i + 2], v[i + 3], s);
#pragma unroll
        for (int j = 0; j < 4; ++j) p.v_cache[page + (d0 + i + j) * 16 + t] = (uint8_t)(w >> (8 * j));
      }
      if (d0 == 0) p.v_scale[(p16 * p.n_kv + kvh) * 16 + t] = s;
    }
    return;
  }
  // ------------------------------------------------------------ NVFP4 caches
  const int bs = p.bs;
  const int64_t page = slot / bs;
  const int t = (int)(slot - page * bs);
  uint8_t *base;
  int sl;
  bool has_gs = true;
  float gs_inv;
  if (is_ik) {
    if (page >= p.idx_pages) {
      if (d0 == 0) set_status(p.status, kDevSlotRange);
      return;
    }
    base = p.idx_cache + page * p.idx_page_bytes;
    sl = 0;
    has_gs = false;
    gs_inv = 1.0f;
  } else {
    if (page >= p.kv_pages) {
      if (d0 == 0) set_status(p.status, kDevSlotRange);
      return;
    }
    base = p.kv_cache + page * p.kv_page_bytes;
    sl = is_k ? 2 * (h - p.k0) : 2 * (h - p.v0) + 1;
    gs_inv = is_k ? p.k_gs_inv : p.v_gs_inv;
  }
  uint8_t *slot_base = base + (int64_t)sl * bs * 72;
  // groups of 16 dims = 4 quads; a group spans 16 / E lanes when E < 16
#pragma unroll
  for (int q0 = 0; q0 < (E >= 16 ? E / 4 : 1); q0 += (E >= 16 ? 4 : 1)) {
    float gmax = 0.f;
    constexpr int QPG = E >= 16 ? 4 : E / 4;  // quads of this group in this thread
#pragma unroll
    for (int q = 0; q < QPG; ++q)
#pragma unroll
      for (int j = 0; j < 4; ++j) gmax = fmaxf(gmax, fabsf(v[4 * (q0 + q) + j]));
    if constexpr (E < 16) {
#pragma unroll
      for (int o = 1; o < 16 / E; o <<= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
    }
    float r;
    const uint8_t sf = nvfp4_scale(gmax, has_gs, gs_inv, r);
    if constexpr (QPG == 4) {  // the group's 16 codes: 8 contiguous bytes, one store
      const int d = d0 + 4 * q0;
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) w[q] = nvfp4_quad(&v[4 * (q0 + q)], r);
      *reinterpret_cast<uint2 *>(slot_base + t * 64 + (d >> 6) * 32 + ((d & 63) >> 1)) =
          make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
    } else {
#pragma unroll
      for (int q = 0; q < QPG; ++q) {
        const int d = d0 + 4 * (q0 + q);
        const uint16_t w = nvfp4_quad(&v[4 * (q0 + q)], r);
        *reinterpret_cast<uint16_t *>(slot_base + t * 64 + (d >> 6) * 32 + ((d & 63) >> 1)) = w;
      }
    }
    const int dg = d0 + 4 * q0;  // first dim of the group part held here
    if ((dg & 15) == 0) {
      const int g = dg >> 4;
      const int off = is_v ? ((t >> 2) * 4 + (g >> 1)) * 8 + (g & 1) * 4 + (t & 3) : t * 8 + g;
      slot_base[bs * 64 + off] = sf;
    }
  }
}

// Signal mode ("vllm.models.minimax_m3.amd.mono.kernels.pre_attn",
// emit_pre_attn.publish_done and emit_k1's done flags): once the (token,
// head) row's stores (outputs and cache bytes) are made, its done word
// done[m * n_heads + head] is set to done_epoch with release semantics at
// GPU scope, so a consumer that reads the epoch there with an acquire load
// then sees every byte of that row.  E < 128 (a warp per row): each lane
// fences its own stores, the warp synchronises, lane 0 releases.  E = 128 (a
// thread per row): the release orders the thread's own stores.
template <int E>
__device__ __forceinline__ void publish_done(const Params &p, const HeadCtx &hc, int d0) {
  if (!p.done) return;
  uint32_t *w = p.done + (int64_t)hc.m * p.n_heads + hc.head;
  if constexpr (E < kHeadDim) {
    __threadfence();
    __syncwarp();
    if (d0 == 0) asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(w), "r"(p.done_epoch) : "memory");
  } else {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(w), "r"(p.done_epoch) : "memory");
  }
}

// The epilogue of one head row, then its done word (when asked for).
template <int E, int CF = -1>
__device__ __forceinline__ void head_epilogue(const Params &p, const HeadCtx &hc, float (&v)[E], int d0) {
  head_epilogue_stores<E, CF>(p, hc, v, d0);
  publish_done<E>(p, hc, d0);
}

// The FP8 V rows of a whole warp, a thread a row (the tensor-core epilogues).
// Every lane of the warp calls it (the warp's head is a V head; `live`:
// the lane holds a token row).  Each lane takes its row's scale and codes
// exactly as head_epilogue_stores does; the cache bytes then leave 8 rows x
// 4 dims an instruction: lane l stores dim 4k + l % 4 of row 8b + l / 4,
// fetched with one shuffle of the row's code word k.  A V page keeps a dim's
// 16 tokens together ([128 dims][16 tokens] bytes), so those 32 bytes fall in
// one 128-byte line of each page the 8 rows touch, where a store of one dim
// for 32 rows touched a line per page of all 32.  Done words (signal mode)
// follow every lane's stores.
__device__ __forceinline__ void v_rows_fp8_warp(const Params &p, const HeadCtx &hc, float (&v)[kHeadDim], bool live) {
  const int lane = threadIdx.x & 31;
  const int kvh = hc.head - p.v0;
  int64_t off = -1;  // byte offset of the row's (page, token) in the V cache; -1: nothing to store
  float s = 1.0f;
  if (live && hc.slot >= 0) {
    const int64_t p16 = page16_of(hc.slot, p.kps);
    if (p16 >= p.num_pages16) {
      set_status(p.status, kDevSlotRange);
    } else {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < kHeadDim; ++i) amax = fmaxf(amax, fabsf(v[i]));
      s = p.static_kv ? 1.0f : (amax == 0.f ? 1.0f : __fdiv_rn(amax, kFp8Max));
      off = (p16 * p.n_kv + kvh) * 2048 + (hc.slot & 15);
    }
  }
  const float rs = __frcp_rn(s);
  int64_t o[4];  // offsets of the rows this lane stores for: 8b + lane / 4
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int src = 8 * b + (lane >> 2);
    o[b] = (int64_t)(((uint64_t)__shfl_sync(0xffffffffu, (uint32_t)((uint64_t)off >> 32), src) << 32) |
                     __shfl_sync(0xffffffffu, (uint32_t)(uint64_t)off, src));
  }
  uint8_t *dst = p.v_cache + 16 * (lane & 3);
  const int sh = 8 * (lane & 3);
#pragma unroll
  for (int k = 0; k < 32; ++k) {  // the row's codes of dims 4k .. 4k + 3, made just before they go out
    uint32_t w = 0u;
    if (off >= 0) {
      bool ok = true;
      w = e4m3x4_prod_checked(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3], rs, ok);
      if (__builtin_expect(!ok, 0)) w = e4m3x4_div(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3], s);
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t x = __shfl_sync(0xffffffffu, w, 8 * b + (lane >> 2));
      if (o[b] >= 0) dst[o[b] + 64 * k] = (uint8_t)(x >> sh);
    }
  }
  if (off >= 0) p.v_scale[(off >> 11) * 16 + (off & 15)] = s;
  if (p.done) {
    __threadfence();
    __syncwarp();
    if (live)
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.done + (int64_t)hc.m * p.n_heads + hc.head),
                   "r"(p.done_epoch)
                   : "memory");
  }
}

}  // namespace pa
