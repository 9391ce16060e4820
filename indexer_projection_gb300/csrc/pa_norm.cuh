// Row normalisation of the pre-attention step (the prologue kernel):
//   acc = ar + res (f32), residual = bf16(acc)
//   n = acc * rsqrt(mean(acc^2) + eps) * (1 + g_in)            (Gemma RMSNorm)
//   per-channel format: s = amax(n) / 448 (1 if 0), xq = e4m3(n / s), a true
//     f32 divide ("vllm.models.minimax_m3.amd.mono.kernels.pre_attn",
//     emit_pre_attn / norm_quant)
//   MXFP8 format: per 32-element block an E8M0 exponent e, the smallest with
//     448 * 2^e >= amax(block), xq = e4m3(n * 2^-e); the scale codes go to
//     the F8_128x4 layout ("vllm.models.minimax_m3.nvidia.ops.
//     qkv_index_fused_epilogue", prepare_SF).
// The normalised row is rounded to f32 once, from an (almost) exact value:
// an activation code that moved by one step would shift the whole token's
// projection, so n (and everything quantised from it) follows the definition
// rather than one particular rounding order.
#pragma once

#include "pa_device.cuh"

namespace pa {

// Error-free transformations (Knuth two-sum, FMA two-product): a + b = s + e
// and a * b = p + e exactly.  Explicit _rn intrinsics keep the compiler from
// contracting or reassociating them.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
__device__ __forceinline__ void two_prod(float a, float b, float &p, float &e) {
  p = __fmul_rn(a, b);
  e = __fmaf_rn(a, b, -p);
}
// (hi, lo) double-float accumulation of sum(acc^2): each square is exact as
// a pair and the running sum carries its rounding error, so the total is
// exact to about 2^-48 whatever the summation order.
__device__ __forceinline__ void dd_add(float &hi, float &lo, float x, float xl) {
  float s, e;
  two_sum(hi, x, s, e);
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(e, xl));
}
// rstd = 1 / sqrt(sum / H + eps) from the block's (hi, lo) partial sums, as
// an unevaluated f32 pair rh + rl accurate to about 2^-44 relative (no FP64:
// it is slow on this part).  The warps' partials are combined by every warp
// with the same shuffle tree (no second barrier, no serial loop over the
// warps).  sum / H and + eps are carried as double-floats; rsqrtf gives r0,
// and one Newton step with its second-order term, r = r0 (1 - t/2 + 3t^2/8)
// with t = x r0^2 - 1 evaluated with FMAs, gives the rest.  Every thread ends
// with the same pair.
// The rstd pair from the row's sum of squares (sh, sl), as described below.
__device__ __forceinline__ void rstd_from_dd(float sh, float sl, int H, float eps, float &rh, float &rl) {
  // x = sum / H + eps
  const float fh = (float)H;
  const float inv = __frcp_rn(fh);
  // sum / H as qh + ql: qh within two ulps of sh / H, the remainder
  // sh - qh * H from one FMA (a few ulps of it at worst, itself ~2^-22 of sh),
  // so the pair is good to ~2^-46 without a divide
  const float qh = __fmul_rn(sh, inv);
  const float rem = __fmaf_rn(-qh, fh, sh);
  const float ql = __fmul_rn(__fadd_rn(rem, sl), inv);
  float xh, xe;
  two_sum(qh, eps, xh, xe);
  const float xl = __fadd_rn(ql, xe);
  const float r0 = rsqrtf(xh);
  float p, pe;
  two_prod(r0, r0, p, pe);
  float t = __fmaf_rn(xh, p, -1.0f);
  t = __fmaf_rn(xh, pe, t);
  t = __fmaf_rn(xl, p, t);
  rh = r0;
  rl = __fmul_rn(__fmul_rn(r0, t), __fmaf_rn(0.375f, t, -0.5f));
}

template <int NTHR>
__device__ __forceinline__ void block_rstd_dd(float hi, float lo, float2 *red, int H, float eps, float &rh,
                                              float &rl) {
  static_assert(NTHR / 32 <= 32 && (NTHR & (NTHR - 1)) == 0, "one warp combines the warps' partials");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, hi, o), ol = __shfl_xor_sync(0xffffffffu, lo, o);
    dd_add(hi, lo, oh, ol);
  }
  if (lane == 0) red[warp] = make_float2(hi, lo);
  __syncthreads();
  constexpr int W = NTHR / 32;
  float2 w = lane < W ? red[lane] : make_float2(0.f, 0.f);
  float sh = w.x, sl = w.y;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    if (o < W) {
      const float oh = __shfl_xor_sync(0xffffffffu, sh, o), ol = __shfl_xor_sync(0xffffffffu, sl, o);
      dd_add(sh, sl, oh, ol);
    }
  }
  sh = __shfl_sync(0xffffffffu, sh, 0);  // lanes >= W summed only zeros
  sl = __shfl_sync(0xffffffffu, sl, 0);
  rstd_from_dd(sh, sl, H, eps, rh, rl);
}

// The smallest e with 448 * 2^e >= amax (amax > 0), clamped to [-127, 127];
// exact, from the bits of amax: amax = (1 + f) 2^E and 448 = 1.75 * 2^8.
__device__ __forceinline__ int mx_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  const uint32_t b = __float_as_uint(amax);
  const int E = (int)((b >> 23) & 255);
  if (E == 0) return -127;
  const int e = (E - 127) - 8 + ((b & 0x7fffffu) > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}
__device__ __forceinline__ float pow2_neg(int e) {  // 2^-e, e in [-127, 127]
  return e == 127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(127 - e) << 23);
}

// 8 elements of a row: acc = ar + res in f32, their bf16 residual bits, and
// the (hi, lo) running sum of acc^2.
__device__ __forceinline__ void acc8(uint4 a, uint4 r, float (&acc)[8], uint4 &resid, float &ss, float &ss_lo) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, rw[4] = {r.x, r.y, r.z, r.w};
  uint32_t ow[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo = bf16_to_f32(aw[i] & 0xffff) + bf16_to_f32(rw[i] & 0xffff);
    float hi = bf16_to_f32(aw[i] >> 16) + bf16_to_f32(rw[i] >> 16);
    acc[2 * i] = lo;
    acc[2 * i + 1] = hi;
    ow[i] = bf16x2_bits(lo, hi);
    float q, ql;
    two_prod(lo, lo, q, ql);
    dd_add(ss, ss_lo, q, ql);
    two_prod(hi, hi, q, ql);
    dd_add(ss, ss_lo, q, ql);
  }
  resid = make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

// The normalised row n = acc * rstd * (1 + gamma), rounded to f32 once from
// an (almost) exact value: rstd as the pair rh + rl, the products as
// error-free pairs.  An FP8 code that moved by one step would shift the whole
// token's projection, so the f32 n (and everything quantised from it)
// follows the definition exactly rather than one particular rounding order.
// In place on 8 elements; gw4 holds their 8 bf16 gammas.
__device__ __forceinline__ void norm8(float (&acc)[8], uint4 gw4, float rh, float rl) {
  const uint32_t gw[4] = {gw4.x, gw4.y, gw4.z, gw4.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float gam = bf16_to_f32(i & 1 ? gw[i >> 1] >> 16 : gw[i >> 1] & 0xffff);
    // acc * (rh + rl) = p + e1 + e2, then (p + e) * (1 + gam)
    float p1, e1, a1, a2, s1, s2;
    two_prod(acc[i], rh, p1, e1);
    const float e = __fadd_rn(e1, __fmul_rn(acc[i], rl));
    two_prod(p1, gam, a1, a2);
    two_sum(p1, a1, s1, s2);
    const float tail = __fadd_rn(__fadd_rn(s2, a2), __fmaf_rn(e, gam, e));
    acc[i] = __fadd_rn(s1, tail);
  }
}

// Per-token FP8: e4m3(n / s), a true f32 divide.
__device__ __forceinline__ uint2 quant8_ptpc(const float (&n)[8], float s) {
  uint2 w;
  w.x = e4m3x4(__fdiv_rn(n[0], s), __fdiv_rn(n[1], s), __fdiv_rn(n[2], s), __fdiv_rn(n[3], s));
  w.y = e4m3x4(__fdiv_rn(n[4], s), __fdiv_rn(n[5], s), __fdiv_rn(n[6], s), __fdiv_rn(n[7], s));
  return w;
}
// MXFP8: e4m3(n * 2^-e), an exact scaling by a power of two.
__device__ __forceinline__ uint2 quant8_mx(const float (&n)[8], float inv) {
  uint2 w;
  w.x = e4m3x4(n[0] * inv, n[1] * inv, n[2] * inv, n[3] * inv);
  w.y = e4m3x4(n[4] * inv, n[5] * inv, n[6] * inv, n[7] * inv);
  return w;
}
// The per-channel scale without a second pass over n: n = acc * rstd *
// (1 + gam) is rounded monotonically and rstd is common to the row, so
// max |n| is the row's maximum of |acc * (1 + gam)| times rstd, rounded once.
// The products are kept as pairs hi + lo (hi = RN, relative error ~2^-46) and
// compared on (hi, lo) in order; amax_from_pair rounds the pair times the
// rstd pair to f32 like norm8 does.
__device__ __forceinline__ void pair_max(float &mh, float &ml, float h, float l) {
  if (h > mh || (h == mh && l > ml)) {
    mh = h;
    ml = l;
  }
}
__device__ __forceinline__ void absprod_max8(const float (&acc)[8], uint4 gw4, float &mh, float &ml) {
  const uint32_t gw[4] = {gw4.x, gw4.y, gw4.z, gw4.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float gam = bf16_to_f32(i & 1 ? gw[i >> 1] >> 16 : gw[i >> 1] & 0xffff);
    float a1, a2, s1, s2;
    two_prod(acc[i], gam, a1, a2);
    two_sum(acc[i], a1, s1, s2);  // acc * (1 + gam) = s1 + s2 + a2
    const float lo = __fadd_rn(s2, a2);
    const float h = __fadd_rn(s1, lo);
    const float l = __fsub_rn(lo, __fsub_rn(h, s1));
    pair_max(mh, ml, fabsf(h), h < 0.f ? -l : l);
  }
}
__device__ __forceinline__ float amax_from_pair(float mh, float ml, float rh, float rl) {
  float q, e;
  two_prod(mh, rh, q, e);
  return __fadd_rn(q, __fmaf_rn(mh, rl, __fmaf_rn(ml, rh, e)));
}
// The block's maximum pair (every thread gets it); red: NTHR / 32 entries.
template <int NTHR>
__device__ __forceinline__ void block_pair_max(float &mh, float &ml, float2 *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float qh = __shfl_xor_sync(0xffffffffu, mh, o), ql = __shfl_xor_sync(0xffffffffu, ml, o);
    pair_max(mh, ml, qh, ql);
  }
  __syncthreads();  // red may still be read by a previous reduction
  if (lane == 0) red[warp] = make_float2(mh, ml);
  __syncthreads();
  mh = red[0].x;
  ml = red[0].y;
#pragma unroll
  for (int w = 1; w < NTHR / 32; ++w) pair_max(mh, ml, red[w].x, red[w].y);
}
__device__ __forceinline__ float amax8(const float (&n)[8]) {
  float a = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(n[e]));
  return a;
}

// ------------------------------------------------ fast path with a check
// The exact n above costs ~17 instructions an element, the true divide of
// the per-channel quantiser ~10 more: at the tensor-core path's thousands of
// rows that makes the prologue instruction-bound.  Only the FP8 codes and
// the scales leave the prologue, so it first computes them from a cheap n
// (t = RN(RN(acc * f) * RN(1 + gamma)), f = RN(rh + rl): within 4 * 2^-24 of
// n, relative) and keeps a result only where every value within a relative
// kSafe of it gives the same code (or MXFP8 block exponent); there the exact
// n must give it too.  Elsewhere (about one element in 2^16) it recomputes
// exactly.  (The per-channel scale needs no check: it comes from the row's
// max |acc (1 + gamma)| times rstd, rounded once; see absprod_max8.)
constexpr float kSafe = 0x1p-20f;  // > 4 * 2^-24 (t) + 2 * 2^-24 (the reciprocal of s)

__device__ __forceinline__ void napprox8(const float (&acc)[8], uint4 gw4, float f, float (&t)[8]) {
  const uint32_t gw[4] = {gw4.x, gw4.y, gw4.z, gw4.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float g1 = __fadd_rn(1.0f, bf16_to_f32(i & 1 ? gw[i >> 1] >> 16 : gw[i >> 1] & 0xffff));
    t[i] = __fmul_rn(__fmul_rn(acc[i], f), g1);
  }
}
// e4m3 codes of 8 values q = t * k, and whether each code is the same for
// every value within a relative kSafe of q.
__device__ __forceinline__ bool codes8_checked(const float (&t)[8], float k, uint2 &w) {
  float q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = __fmul_rn(t[i], k);
  const float lo = 1.0f - kSafe, hi = 1.0f + kSafe;
  w.x = e4m3x4(q[0], q[1], q[2], q[3]);
  w.y = e4m3x4(q[4], q[5], q[6], q[7]);
  const uint32_t l0 = e4m3x4(q[0] * lo, q[1] * lo, q[2] * lo, q[3] * lo), l1 = e4m3x4(q[4] * lo, q[5] * lo, q[6] * lo, q[7] * lo);
  const uint32_t h0 = e4m3x4(q[0] * hi, q[1] * hi, q[2] * hi, q[3] * hi), h1 = e4m3x4(q[4] * hi, q[5] * hi, q[6] * hi, q[7] * hi);
  return (w.x == l0) & (w.x == h0) & (w.y == l1) & (w.y == h1);
}

// Normalise and quantise token row m with the NTHR threads of the block
// (every thread must call it).  Chunks of 8 elements: thread tid holds chunks
// tid + NTHR * j, j < MAXC, so H <= 8 * NTHR * MAXC; NTHR % 4 == 0 keeps the
// four chunks of a 32-element MXFP8 block in lanes 4i .. 4i + 3.
template <int WFMT, int NTHR, int MAXC>
__device__ __forceinline__ void norm_quant_row(const Params &p, const int m, float2 *red2) {
  static_assert(NTHR % 32 == 0, "whole warps");
  const int tid = threadIdx.x;
  const int H = p.H, nch = H >> 3, ksf = H >> 5;
  const uint4 *ar = reinterpret_cast<const uint4 *>(p.ar + (int64_t)m * H);
  const uint4 *res = reinterpret_cast<const uint4 *>(p.res + (int64_t)m * H);
  uint4 *rout = p.residual ? reinterpret_cast<uint4 *>(p.residual + (int64_t)m * H) : nullptr;
  float acc[MAXC][8];
  float ss = 0.f, ss_lo = 0.f, mh = 0.f, ml = 0.f;
  uint4 gpre[MAXC];  // the input-norm gamma, loaded with the row
  const uint4 *g4 = reinterpret_cast<const uint4 *>(p.g_in);
#pragma unroll
  for (int j = 0; j < MAXC; ++j) {
    const int c = tid + NTHR * j;
    if (c < nch) gpre[j] = __ldg(g4 + c);
  }
#pragma unroll
  for (int j = 0; j < MAXC; ++j) {
    const int c = tid + NTHR * j;
    if (c < nch) {
      uint4 rb;
      acc8(__ldcs(ar + c), __ldcs(res + c), acc[j], rb, ss, ss_lo);
      if (rout) __stcs(rout + c, rb);
      if (WFMT == 0) absprod_max8(acc[j], gpre[j], mh, ml);
    }
  }
  float rh, rl;
  block_rstd_dd<NTHR>(ss, ss_lo, red2, H, p.eps, rh, rl);
  const float f = __fadd_rn(rh, rl);
  uint2 *xq = reinterpret_cast<uint2 *>(p.xq + (int64_t)m * H);
  if (WFMT == 0) {
    // the scale s = amax(n) / 448: the row's max |acc (1 + gamma)| times rstd
    block_pair_max<NTHR>(mh, ml, red2);
    const float tmax = amax_from_pair(mh, ml, rh, rl);
    const float s = tmax == 0.f ? 1.0f : __fdiv_rn(tmax, kFp8Max);
    const float rs = __frcp_rn(s);
#pragma unroll
    for (int j = 0; j < MAXC; ++j) {
      const int c = tid + NTHR * j;
      if (c < nch) {
        float t[8];
        napprox8(acc[j], gpre[j], f, t);
        uint2 w;
        if (!codes8_checked(t, rs, w) || p.exact_norm) {  // near a code boundary: exact n and a true divide
          norm8(acc[j], gpre[j], rh, rl);
          w = quant8_ptpc(acc[j], s);
        }
        xq[c] = w;
      }
    }
    if (tid == 0) p.x_scale[m] = s;
  } else {
    // a 32-element block is 4 consecutive chunks, held by lanes 4i .. 4i + 3
#pragma unroll
    for (int j = 0; j < MAXC; ++j) {
      const int c = tid + NTHR * j;
      if (j * NTHR < nch) {  // warp-uniform: every lane reaches the shuffles
        float t[8];
        float bm = 0.f;
        if (c < nch) {
          napprox8(acc[j], gpre[j], f, t);
          bm = amax8(t);
        }
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
        // the exponent is exact where every amax within kSafe gives it
        const bool e_ok = mx_exponent(bm * (1.0f - kSafe)) == mx_exponent(bm * (1.0f + kSafe)) && !p.exact_norm;
        const bool exact = __any_sync(0xffffffffu, !e_ok);  // warp-uniform
        if (exact) {  // rare: this warp's blocks from the exact n (acc[j] becomes n)
          if (c < nch) {
            norm8(acc[j], gpre[j], rh, rl);
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = acc[j][i];
          }
          bm = c < nch ? amax8(t) : 0.f;
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
        }
        if (c < nch) {
          const int e = mx_exponent(bm);
          uint2 w;
          if (!codes8_checked(t, pow2_neg(e), w) || p.exact_norm) {  // near a code boundary: from the exact n
            if (!exact) norm8(acc[j], gpre[j], rh, rl);
            w = quant8_mx(acc[j], pow2_neg(e));
          }
          xq[c] = w;
          if ((c & 3) == 0) p.xsf[sf128x4_offset(m, c >> 2, ksf)] = (uint8_t)(e + 127);
        }
      }
    }
  }
}

}  // namespace pa
