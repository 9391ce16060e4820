// The DSpark drafter's attention ("vllm.models.minimax_m3.amd.mono.drafter.
// attention": module summary, qkv_rows, window, kv_load, block_math /
// block_acc, store_partial, merge_task), as three kernels.
//
// pa_drafter_qkv_kernel (qkv_rows): a warp a (row, head) of the drafter's
// projection rows: Gemma head RMSNorm and partial NeoX RoPE for the 16 q heads
// and k, then E4M3 (unit scale): q into the q8 rows the attention reads, k and
// v into the drafter cache at the row's slot.
//
// pa_drafter_attn_kernel: a CTA a (partition, request).  The page runs a wave
// a query row over 16 heads with the keys as the MMA's rows; here the whole
// request is one 128-row MMA tile (row 16 j + h = head h of query row j, up to
// 8 rows, 7 on the page), so each 128-key block is two 128 x 128 x 128 FP8
// tcgen05 MMAs:
//   S = Q K^T   (A: the request's q8 rows, B: the block's K bytes, both
//               K-major, 128-byte swizzle, loaded by TMA straight from the
//               cache's 256-byte key records)
//   O += P V    (A: E4M3(P) written by the softmax threads into a swizzled
//               shared tile, B: the block's V bytes as loaded, i.e. MN-major:
//               a key's 128 dims are contiguous)
// with S and O in tensor memory (256 columns, two CTAs an SM).  Four softmax
// warps own a row each per thread (TMEM lane = row): they read the row's 128
// scores in one round trip (S is then free, so the next block's QK^T runs
// while they work), take the block's masked row maximum, alpha, P = exp2(s C
// - (m C - 8)) (P x 256 at the new maximum), l, the E4M3 codes of P (written
// straight into the P tile once the previous PV is done), and rescale O by
// alpha in tensor memory before this block's PV.  One thread issues the TMA
// copies (two stages of K + V), one the MMAs.
// Keys outside [lo, hi] of a window-edge block hold whatever the cache held
// (stale or never written bytes, possibly E4M3 NaN codes): their scores are
// masked and their V rows zeroed in shared memory before the PV MMA, as the
// page's kv_load zeroes them.
// Each partition stores (m, l, o) of its rows (store_partial).
//
// pa_drafter_merge_kernel (merge_task): a CTA a query row, a thread a (head,
// 16 dims): the request's partitions merged in order, rounded to bf16 and
// quantised to MXFP8 (a 32-dim block is two neighbouring threads).  It waits
// for the attention kernel through programmatic dependent launch, so the
// whole merge runs spread over the GPU instead of on one CTA a request.
//
// Every wait is bounded (PA_DEV_WAIT_TIMEOUT); a block id outside the cache,
// or a window block past the block table, is read as zeros, masked and
// flagged (PA_DEV_SLOT_RANGE).
#include <cstdint>

#include <cuda_bf16.h>

#include "../../include/pre_attn.h"
#include "pa_device.cuh"
#include "pa_launch.h"
#include "pa_tc.cuh"
#include "pa_tma.h"

namespace pa {
namespace {

constexpr int kDaHeads = 16;
constexpr int kDaMaxRows = 8;             // query rows a request: 16 heads x 8 = 128 MMA rows
constexpr int kDaKeyBytes = 256;          // a key's K bytes, then its V bytes
constexpr int kDaTile = 128 * 128;        // a 128 x 128-byte operand tile
constexpr int kDaStages = 2;              // K + V stages
constexpr int kDaThreads = 192;           // warp 0 TMA, warp 1 MMA + TMEM, warps 2..5 softmax
constexpr uint32_t kDaTmemCols = 256;     // S at column 0, O at column 128
constexpr int kDaOCol = 128;
// a partition's (m, l, o): m[128], l[128] f32, then o as [32 dim quads][128 rows] float4 (a row's
// quad q at float4 index 128 q + row: the threads of a row each store 16 contiguous bytes a quad)
constexpr int64_t kDaPartBytes = 2 * 128 * 4 + 128 * 128 * 4;
constexpr int kDaQkvThreads = 256;

// shared memory (from a 1024-byte aligned base)
constexpr int kSmQ = 0;
constexpr int kSmP = kSmQ + kDaTile;
constexpr int kSmK = kSmP + kDaTile;
constexpr int kSmV = kSmK + kDaStages * kDaTile;
constexpr int kSmBars = kSmV + kDaStages * kDaTile;
constexpr int kDaSmem = kSmBars + 256 + 1024;  // + barriers, + alignment slack

constexpr uint32_t kIdescQK = idesc_f8(128, 128);
constexpr uint32_t kIdescPV = idesc_f8(128, 128) | (1u << 16);  // B (V) MN-major

// Descriptor of V as an MN-major operand: rows of 128 bytes (a key's 128 dims,
// one swizzle atom wide, so there is no second atom along N), 128-byte
// swizzle, 8-key groups 1024 bytes apart.  The leading-byte offset is set to
// the same 1024 bytes: with a single atom along N it only ever describes the
// K-direction stride, whichever of the two fields the layout reads for it.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(1024 >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// 2^x on the SFU (ex2.approx: relative error a few ulp; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct QkvParams {
  const __nv_bfloat16 *qkv;
  int64_t qkv_stride;
  const __nv_bfloat16 *qn, *kn;
  float eps;
  const __nv_bfloat16 *cos_sin;
  int64_t max_pos;
  const int64_t *positions, *slot_mapping;
  uint8_t *cache;
  int64_t num_blocks;
  uint8_t *q8;
  int M;
  uint32_t *status;
};

struct AttnParams {
  const int32_t *block_table;
  const int32_t *seq_lens;
  const int64_t *positions;
  int64_t num_blocks;
  int R, q_len, bt_width, window, max_blocks, part_blocks, maxp;
  float C;  // sm_scale * log2(e)
  uint8_t *parts;
  __nv_bfloat16 *out_bf16;
  uint8_t *out_codes, *out_scales;
  uint32_t *status;
  int test_timeout;
};

// --------------------------------------------------------------- kernel 1
__global__ void __launch_bounds__(kDaQkvThreads) pa_drafter_qkv_kernel(QkvParams a, int use_pdl) {
  if (use_pdl) {
    pdl_wait();  // the projection rows come from the previous kernel
    pdl_trigger();
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t task = (int64_t)blockIdx.x * (kDaQkvThreads / 32) + warp;
  if (task >= (int64_t)a.M * (kDaHeads + 2)) return;
  const int m = (int)(task / (kDaHeads + 2)), h = (int)(task % (kDaHeads + 2));
  const int d0 = 4 * lane;
  const uint2 raw = *reinterpret_cast<const uint2 *>(a.qkv + (int64_t)m * a.qkv_stride + h * kHeadDim + d0);
  float v[4] = {bf16_to_f32(raw.x & 0xffff), bf16_to_f32(raw.x >> 16), bf16_to_f32(raw.y & 0xffff),
                bf16_to_f32(raw.y >> 16)};
  if (h <= kDaHeads) {  // q heads and k: head norm, RoPE
    int64_t pos = ld_i64(a.positions + m);
    if (pos < 0 || pos >= a.max_pos) {
      if (lane == 0) set_status(a.status, kDevPosRange);
      pos = pos < 0 ? 0 : a.max_pos - 1;
    }
    head_rmsnorm<4>(v, d0, h < kDaHeads ? a.qn : a.kn, a.eps);
    head_rope<4>(v, d0, a.cos_sin + pos * kRotDim);
  }
  const uint32_t w = e4m3x4(v[0], v[1], v[2], v[3]);
  if (h < kDaHeads) {
    *reinterpret_cast<uint32_t *>(a.q8 + ((int64_t)m * kDaHeads + h) * kHeadDim + d0) = w;
    return;
  }
  const int64_t slot = ld_i64(a.slot_mapping + m);
  if (slot < 0) return;
  if (slot >= a.num_blocks * 128) {
    if (lane == 0) set_status(a.status, kDevSlotRange);
    return;
  }
  *reinterpret_cast<uint32_t *>(a.cache + slot * kDaKeyBytes + (h - kDaHeads) * kHeadDim + d0) = w;
}

// --------------------------------------------------------------- kernel 2
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// The request's window (window): keys lo .. hi, from the first row's window
// start, below seq_len, at most max_blocks blocks from lo's.
struct Window {
  int64_t p0, lo, hi;
  int b_lo, nblk;  // first block, blocks (<= 0: none)
};
__device__ __forceinline__ Window request_window(const AttnParams &a, int r) {
  Window w;
  w.p0 = ld_i64(a.positions + (int64_t)r * a.q_len);
  const int64_t seq = __ldg(a.seq_lens + r);
  w.lo = w.p0 - (a.window - 1);
  if (w.lo < 0) w.lo = 0;
  w.hi = (w.lo / 128 + a.max_blocks) * 128 - 1;
  if (seq - 1 < w.hi) w.hi = seq - 1;
  w.b_lo = (int)(w.lo / 128);
  w.nblk = w.hi < w.lo ? 0 : (int)(w.hi / 128) - w.b_lo + 1;
  return w;
}

// Physical block of window block b (-1: past the block table or outside the cache).
__device__ __forceinline__ int64_t phys_block(const AttnParams &a, int r, int b) {
  if (b >= a.bt_width) return -1;
  const int64_t phys = __ldg(a.block_table + (int64_t)r * a.bt_width + b);
  return phys < 0 || phys >= a.num_blocks ? -1 : phys;
}

// The smallest power-of-two exponent e with 448 * 2^e >= amax (E8M0 range).
__device__ __forceinline__ int mx_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  const uint32_t b = __float_as_uint(amax);
  const int eb = (int)(b >> 23);
  if (eb == 0) return -127;  // below 2^-126: 448 * 2^-127 covers it
  // amax = 1.f * 2^(eb - 127); 448 = 1.75 * 2^8
  int e = (b & 0x7fffff) <= 0x600000u ? eb - 127 - 8 : eb - 127 - 7;
  return e < -127 ? -127 : e > 127 ? 127 : e;
}

__global__ void __launch_bounds__(kDaThreads, 2)
    pa_drafter_attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                           AttnParams a, int use_pdl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t *kv_full = reinterpret_cast<uint64_t *>(smem + kSmBars);
  uint64_t *kv_empty = kv_full + kDaStages;
  uint64_t *q_full = kv_empty + kDaStages;
  uint64_t *s_full = q_full + 1;   // S of the block written (MMA commit)
  uint64_t *s_free = s_full + 1;   // S read by the 4 softmax warps
  uint64_t *p_full = s_free + 1;   // P written, O rescaled (4 softmax warps)
  uint64_t *o_done = p_full + 1;   // the block's PV MMA done (MMA commit)
  uint64_t *never = o_done + 1;    // testing: nothing arrives on it
  uint64_t *drain = never + 1;     // the MMA issuer's last commit on an abnormal exit
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int part = blockIdx.x, r = blockIdx.y;
  const uint64_t lim = a.test_timeout ? kTestWaitNs : kWaitNs;

  if (tid == 0) {
    for (int s = 0; s < kDaStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(never, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmKV)) : "memory");
  }
  if (use_pdl) pdl_wait();  // q8 and the new keys come from the previous kernel
  const Window win = request_window(a, r);
  const int na = (win.nblk + a.part_blocks - 1) / a.part_blocks;
  if (part >= na) return;  // no partition here (no key at all: the merge writes zero rows)
  const int b0 = win.b_lo + part * a.part_blocks;
  const int nb = min(a.part_blocks, win.nblk - part * a.part_blocks);

  if (warp == 1) tc_alloc(tmem_slot, kDaTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      int last_ph[kDaStages] = {-1, -1};  // phase each stage was last loaded with
      mbar_expect_tx(q_full, kDaTile);
      tma_tile(smem_u32(smem + kSmQ), &tmQ, 0, r * kDaHeads * a.q_len, q_full);
      for (int t = 0; t < nb; ++t) {
        const int s = t % kDaStages;
        const uint32_t ph = (uint32_t)(t / kDaStages) & 1;
        if (!mbar_wait(&kv_empty[s], ph ^ 1, a.status, lim)) {
          ok = false;
          break;
        }
        int64_t phys = phys_block(a, r, b0 + t);
        if (phys < 0) {
          set_status(a.status, kDevSlotRange);
          phys = a.num_blocks;  // rows past the cache: the copy reads zeros
        }
        last_ph[s] = (int)ph;
        mbar_expect_tx(&kv_full[s], 2 * kDaTile);
        tma_tile(smem_u32(smem + kSmK + s * kDaTile), &tmKV, 0, (int)(phys * 128), &kv_full[s]);
        tma_tile(smem_u32(smem + kSmV + s * kDaTile), &tmKV, 128, (int)(phys * 128), &kv_full[s]);
      }
      if (!ok) {  // the copies in flight land before the CTA exits
        mbar_wait(q_full, 0, a.status, lim);
        for (int s = 0; s < kDaStages; ++s)
          if (last_ph[s] >= 0) mbar_wait(&kv_full[s], (uint32_t)last_ph[s], a.status, lim);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    // S of the next block as soon as the softmax threads have read this one
    // (it runs while they work), then this block's PV once its P is written
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0, a.status, lim) && mbar_wait(&kv_full[0], 0, a.status, lim);
      const uint64_t qd = sdesc_sw128(smem_u32(smem + kSmQ));
      const uint64_t pd = sdesc_sw128(smem_u32(smem + kSmP));
      if (ok) {
        tc_fence_after();
        const uint64_t kd = sdesc_sw128(smem_u32(smem + kSmK));
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_f8(tmem, qd + 2 * k, kd + 2 * k, kIdescQK, k > 0);
        tc_commit(s_full);
      }
      for (int t = 0; t < nb && ok; ++t) {
        const int s = t % kDaStages;
        if (t + 1 < nb) {
          const int s1 = (t + 1) % kDaStages;
          if (!mbar_wait(&kv_full[s1], (uint32_t)((t + 1) / kDaStages) & 1, a.status, lim) ||
              !mbar_wait(s_free, (uint32_t)t & 1, a.status, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kd = sdesc_sw128(smem_u32(smem + kSmK + s1 * kDaTile));
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_f8(tmem, qd + 2 * k, kd + 2 * k, kIdescQK, k > 0);
          tc_commit(s_full);
        }
        if (!mbar_wait(p_full, (uint32_t)t & 1, a.status, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // O += P V: 32 keys an MMA; V's 32 key rows are 4096 bytes on (+256 in the
        // descriptor's 16-byte address field), P's 32 bytes along K +2
        const uint64_t vd = sdesc_sw128_mn(smem_u32(smem + kSmV + s * kDaTile));
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_f8(tmem + kDaOCol, pd + 2 * k, vd + 256 * k, kIdescPV, (t | k) != 0);
        tc_commit(o_done);
        tc_commit(&kv_empty[s]);
      }
      if (!ok) {  // the MMAs issued complete before the TMEM is freed
        tc_commit(drain);
        mbar_wait(drain, 0, a.status, lim);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int qd = warp & 3;
    const int row = 32 * qd + lane;  // TMEM lane = S / O row = q8 row 16 j + h
    const int j = row >> 4;
    const bool live = j < a.q_len;
    const uint32_t trow = tmem + ((uint32_t)(32 * qd) << 16);
    const float C = a.C;
    int64_t klo = win.p0 + j - a.window + 1;  // the row's first key
    if (klo < win.lo) klo = win.lo;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    if (a.test_timeout && !mbar_wait(never, 0, a.status, lim)) ok = false;
    for (int t = 0; t < nb && ok; ++t) {
      const int s = t % kDaStages;
      const int64_t kb = (int64_t)(b0 + t) * 128;
      const bool bad = phys_block(a, r, b0 + t) < 0;
      int kmin = 128, kmax = -1;  // valid keys kb + kmin .. kb + kmax of this row
      if (!live) {
        kmin = 0, kmax = 127;  // padding rows: computed, never used
      } else if (!bad) {
        const int64_t x = klo - kb, y = win.hi - kb;
        kmin = x < 0 ? 0 : x > 128 ? 128 : (int)x;
        kmax = y > 127 ? 127 : y < -1 ? -1 : (int)y;
      }
      const bool full = kmin == 0 && kmax == 127;
      if (!mbar_wait(s_full, (uint32_t)t & 1, a.status, lim)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the row's 128 scores in one round trip; S is then free for the next
      // block's QK^T, which runs while this block's exponentials do
      float x[128];
      tc_ld64(trow, *reinterpret_cast<float(*)[64]>(&x[0]));
      tc_ld64(trow + 64, *reinterpret_cast<float(*)[64]>(&x[64]));
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      // window-edge blocks (some row of the warp has keys outside its range):
      // those scores become -inf (P = 2^-inf = 0); the branch is warp-uniform
      if (__any_sync(0xffffffffu, !full)) {
#pragma unroll
        for (int k = 0; k < 128; ++k) x[k] = ((k >= kmin) & (k <= kmax)) ? x[k] : -INFINITY;
      }
      float m4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
      for (int k = 4; k < 128; ++k) m4[k & 3] = fmaxf(m4[k & 3], x[k]);
      const float mb = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      const float mn = fmaxf(m_run, mb);
      const float ms = mn == -INFINITY ? 0.f : mn;
      const float alpha = live ? ex2((m_run - ms) * C) : 1.0f;  // padding rows: no rescale
      const float off = ms * C - 8.0f;
      // the previous block's PV is done: P's tile and O are free
      if (t > 0) {
        if (!mbar_wait(o_done, (uint32_t)(t - 1) & 1, a.status, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      // P (x 256 at the new maximum), its sum, and its E4M3 codes straight
      // into the swizzled P tile, 16 keys a 16-byte chunk
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
      uint8_t *prow = smem + kSmP + row * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float pq[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            pq[u] = ex2(fmaf(x[16 * c + 4 * q + u], C, -off));
            s4[u] += pq[u];
          }
          w[q] = e4m3x4(pq[0], pq[1], pq[2], pq[3]);
        }
        if (live) *reinterpret_cast<uint4 *>(prow + ((c ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      l_run = fmaf(l_run, alpha, (s4[0] + s4[1]) + (s4[2] + s4[3]));
      m_run = mn;
      // O rescaled by alpha before this block's PV accumulates into it
      if (t > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {  // one round trip
        float o[128];
        tc_ld64(trow + kDaOCol, *reinterpret_cast<float(*)[64]>(&o[0]));
        tc_ld64(trow + kDaOCol + 64, *reinterpret_cast<float(*)[64]>(&o[64]));
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 128; ++e) o[e] *= alpha;
        tc_st64(trow + kDaOCol, *reinterpret_cast<const float(*)[64]>(&o[0]));
        tc_st64(trow + kDaOCol + 64, *reinterpret_cast<const float(*)[64]>(&o[64]));
        tc_wait_st();
      }
      // keys of the block outside [lo, hi]: their V rows to zero
      const int64_t key = kb + row;
      if (key < win.lo || key > win.hi) {
        if (!mbar_wait(&kv_full[s], (uint32_t)(t / kDaStages) & 1, a.status, lim)) {
          ok = false;
          break;
        }
        uint4 *vrow = reinterpret_cast<uint4 *>(smem + kSmV + s * kDaTile + row * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) vrow[c] = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // the partition's (m, l, o) of this row (store_partial)
    if (ok && !mbar_wait(o_done, (uint32_t)(nb - 1) & 1, a.status, lim)) ok = false;
    tc_fence_after();
    uint8_t *pp = a.parts + ((int64_t)r * a.maxp + part) * kDaPartBytes;
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
      float o[64];
      tc_ld64(trow + kDaOCol + 64 * hf, o);
      tc_wait_ld();
      if (live) {  // quad-major: a warp's 32 rows of a quad are 512 contiguous bytes
        float4 *dst = reinterpret_cast<float4 *>(pp + 1024) + (16 * hf) * 128 + row;
#pragma unroll
        for (int q = 0; q < 16; ++q) dst[q * 128] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      }
    }
    if (live) {
      reinterpret_cast<float *>(pp)[row] = m_run;
      reinterpret_cast<float *>(pp + 512)[row] = l_run;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (use_pdl) pdl_trigger();
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc(tmem, kDaTmemCols);
  }
}

// ------------------------------------------------------------ kernel 3
// The merge (merge_task): a CTA a query row m = r * q_len + j, a thread a
// (head h, 16 dims); the request's partitions are merged in order:
//   m* = max m_i, w_i = 2^((m_i - m*) C) (0 for a partition without a valid
//   key of the row), out = sum w_i o_i / sum w_i l_i (0 if that sum is 0),
// rounded to bf16, then MXFP8: each 32-dim block (two neighbouring threads)
// takes the smallest E8M0 scale 2^e with 448 * 2^e >= its amax, codes
// E4M3(x * 2^-e).  A request without keys gets zero rows.
constexpr int kDaMergeThreads = 128;
constexpr int kDaMergeBatch = 4;  // partitions whose loads are in flight together

__global__ void __launch_bounds__(kDaMergeThreads) pa_drafter_merge_kernel(AttnParams a, int use_pdl) {
  const int tid = threadIdx.x;
  const int m_row = blockIdx.x;
  const int r = m_row / a.q_len, j = m_row - r * a.q_len;
  const int h = tid >> 3, piece = tid & 7;
  const int row = kDaHeads * j + h;  // the partials' row
  if (use_pdl) pdl_wait();           // the partials come from the attention kernel
  const Window win = request_window(a, r);
  const int na = win.nblk > 0 ? (win.nblk + a.part_blocks - 1) / a.part_blocks : 0;
  const uint8_t *pr = a.parts + (int64_t)r * a.maxp * kDaPartBytes;
  float mst = -INFINITY;
  for (int i0 = 0; i0 < na; i0 += 8) {
    float mi[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      mi[u] = i0 + u < na ? __ldcg(reinterpret_cast<const float *>(pr + (int64_t)(i0 + u) * kDaPartBytes) + row)
                          : -INFINITY;
#pragma unroll
    for (int u = 0; u < 8; ++u) mst = fmaxf(mst, mi[u]);
  }
  float L = 0.f, acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  for (int i0 = 0; i0 < na; i0 += kDaMergeBatch) {
    float mi[kDaMergeBatch], li[kDaMergeBatch];
    float4 oi[kDaMergeBatch][4];
#pragma unroll
    for (int u = 0; u < kDaMergeBatch; ++u) {
      const bool in = i0 + u < na;
      const uint8_t *pi = pr + (int64_t)(in ? i0 + u : 0) * kDaPartBytes;
      mi[u] = in ? __ldcg(reinterpret_cast<const float *>(pi) + row) : -INFINITY;
      li[u] = in ? __ldcg(reinterpret_cast<const float *>(pi + 512) + row) : 0.f;
      const float4 *o = reinterpret_cast<const float4 *>(pi + 1024) + (4 * piece) * 128 + row;
#pragma unroll
      for (int q = 0; q < 4; ++q) oi[u][q] = in ? __ldcg(o + q * 128) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kDaMergeBatch; ++u) {  // in partition order
      if (mi[u] == -INFINITY) continue;          // no valid key of this row there
      const float w = ex2((mi[u] - mst) * a.C);
      L = fmaf(w, li[u], L);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[4 * q] = fmaf(w, oi[u][q].x, acc[4 * q]);
        acc[4 * q + 1] = fmaf(w, oi[u][q].y, acc[4 * q + 1]);
        acc[4 * q + 2] = fmaf(w, oi[u][q].z, acc[4 * q + 2]);
        acc[4 * q + 3] = fmaf(w, oi[u][q].w, acc[4 * q + 3]);
      }
    }
  }
  // out = o / l in bf16, then the MXFP8 block of this thread and its neighbour
  float amax = 0.f;
  uint32_t bw[8];
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const float x0 = L > 0.f ? acc[e] / L : 0.f, x1 = L > 0.f ? acc[e + 1] / L : 0.f;
    const uint32_t h = bf16x2_bits(x0, x1);
    acc[e] = __uint_as_float(h << 16);
    acc[e + 1] = __uint_as_float(h & 0xffff0000u);
    amax = fmaxf(amax, fmaxf(fabsf(acc[e]), fabsf(acc[e + 1])));
    bw[e >> 1] = h;
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  const int e = mx_exponent(amax);
  const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e (e <= 126 for a bf16 amax)
  uint32_t cw[4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    cw[q] = e4m3x4(acc[4 * q] * inv, acc[4 * q + 1] * inv, acc[4 * q + 2] * inv, acc[4 * q + 3] * inv);
  const int col = h * kHeadDim + 16 * piece;
  *reinterpret_cast<uint4 *>(a.out_codes + (int64_t)m_row * 2048 + col) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  if ((piece & 1) == 0) a.out_scales[(int64_t)m_row * 64 + (col >> 5)] = (uint8_t)(e + 127);
  if (a.out_bf16) {
    uint4 *bd = reinterpret_cast<uint4 *>(a.out_bf16 + (int64_t)m_row * 2048 + col);
    bd[0] = make_uint4(bw[0], bw[1], bw[2], bw[3]);
    bd[1] = make_uint4(bw[4], bw[5], bw[6], bw[7]);
  }
  if (use_pdl) pdl_trigger();
}

}  // namespace
}  // namespace pa

extern "C" int pre_attn_drafter_part_blocks(int R, int max_blocks, int num_sms) {
  if (R < 1 || max_blocks < 1 || num_sms < 1) return -PA_ERR_SHAPE;
  // as many partitions a request as keep every partition of every request
  // in one wave of two CTAs an SM, cut evenly
  int per = 2 * num_sms / R;
  if (per < 1) per = 1;
  const int pb = (max_blocks + per - 1) / per;
  return pb < 1 ? 1 : pb > max_blocks ? max_blocks : pb;
}

extern "C" size_t pre_attn_drafter_workspace_bytes(int R, int max_blocks, int part_blocks) {
  if (R < 1 || max_blocks < 1 || part_blocks < 1) return 0;
  const int64_t maxp = (max_blocks + part_blocks - 1) / part_blocks;
  return (size_t)((int64_t)R * maxp * pa::kDaPartBytes);
}

extern "C" int pre_attn_drafter_attention(const pa_drafter_args *in, void *stream) {
  using namespace pa;
  if (!in) return PA_ERR_NULL;
  const pa_drafter_args &x = *in;
  if (!x.positions || !x.cache || !x.block_table || !x.seq_lens || !x.q8 || !x.out_codes || !x.out_scales ||
      !x.workspace || !x.status)
    return PA_ERR_NULL;
  if (x.qkv && (!x.qn || !x.kn || !x.cos_sin || !x.slot_mapping)) return PA_ERR_NULL;
  if (x.R < 0 || x.R > 65535 || x.q_len < 1 || x.q_len > kDaMaxRows || x.bt_width < 1 || x.num_blocks < 1 ||
      x.num_blocks >= (1 << 24))
    return PA_ERR_SHAPE;
  if (x.qkv && (x.qkv_stride < (kDaHeads + 2) * kHeadDim || x.qkv_stride % 8 || x.max_pos < 1)) return PA_ERR_SHAPE;
  if (x.window < 1 || x.max_blocks < 1 || x.max_blocks > 65535 || x.part_blocks < 0 ||
      !(x.sm_scale > 0.f && x.sm_scale < INFINITY) || (x.qkv && !(x.eps >= 0.f)))
    return PA_ERR_CONFIG;
  const uintptr_t a16 = 15;
  auto mis = [](const void *p, uintptr_t m) { return (reinterpret_cast<uintptr_t>(p) & m) != 0; };
  if (mis(x.cache, a16) || mis(x.q8, a16) || mis(x.out_codes, a16) || (x.out_bf16 && mis(x.out_bf16, a16)) ||
      mis(x.workspace, 255) || mis(x.status, 3) || mis(x.positions, 7) || mis(x.block_table, 3) ||
      mis(x.seq_lens, 3))
    return PA_ERR_ALIGN;
  if (x.qkv && (mis(x.qkv, a16) || mis(x.qn, a16) || mis(x.kn, a16) || mis(x.cos_sin, a16) || mis(x.slot_mapping, 7)))
    return PA_ERR_ALIGN;
  if (x.R == 0) return PA_OK;
  int pb = x.part_blocks;
  if (pb == 0) {
    const int sms = current_device_sms();
    if (sms < 1) return record_cuda_error(cudaGetLastError());
    pb = pre_attn_drafter_part_blocks(x.R, x.max_blocks, sms);
  }
  if (pb > x.max_blocks) pb = x.max_blocks;
  if (x.workspace_bytes < pre_attn_drafter_workspace_bytes(x.R, x.max_blocks, pb)) return PA_ERR_WORKSPACE;
  const bool pdl = !(x.flags & PA_FLAG_NO_PDL);
  const int M = x.R * x.q_len;
  const cudaStream_t s = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaError_t e;
  if (x.qkv) {
    QkvParams q;
    q.qkv = static_cast<const __nv_bfloat16 *>(x.qkv);
    q.qkv_stride = x.qkv_stride;
    q.qn = static_cast<const __nv_bfloat16 *>(x.qn);
    q.kn = static_cast<const __nv_bfloat16 *>(x.kn);
    q.eps = x.eps;
    q.cos_sin = static_cast<const __nv_bfloat16 *>(x.cos_sin);
    q.max_pos = x.max_pos;
    q.positions = x.positions;
    q.slot_mapping = x.slot_mapping;
    q.cache = static_cast<uint8_t *>(x.cache);
    q.num_blocks = x.num_blocks;
    q.q8 = static_cast<uint8_t *>(x.q8);
    q.M = M;
    q.status = x.status;
    cudaLaunchConfig_t cfg = {};
    const int64_t warps = (int64_t)M * (kDaHeads + 2);
    cfg.gridDim = dim3((unsigned)((warps + kDaQkvThreads / 32 - 1) / (kDaQkvThreads / 32)));
    cfg.blockDim = dim3(kDaQkvThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, pa_drafter_qkv_kernel, q, pdl ? 1 : 0);
    if (e != cudaSuccess) return record_cuda_error(e);
  }
  CUtensorMap tmQ, tmKV;
  if (!map_rows_sw128(&tmQ, x.q8, (uint64_t)M * kDaHeads, kHeadDim, kHeadDim, 128) ||
      !map_rows_sw128(&tmKV, x.cache, (uint64_t)x.num_blocks * 128, kDaKeyBytes, 128, 128))
    return record_cuda_error(cudaErrorInvalidValue);
  AttnParams p;
  p.block_table = x.block_table;
  p.seq_lens = x.seq_lens;
  p.positions = x.positions;
  p.num_blocks = x.num_blocks;
  p.R = x.R;
  p.q_len = x.q_len;
  p.bt_width = x.bt_width;
  p.window = x.window;
  p.max_blocks = x.max_blocks;
  p.part_blocks = pb;
  p.maxp = (x.max_blocks + pb - 1) / pb;
  p.C = (float)((double)x.sm_scale * 1.4426950408889634);  // log2(e)
  p.parts = static_cast<uint8_t *>(x.workspace);
  p.out_bf16 = static_cast<__nv_bfloat16 *>(x.out_bf16);
  p.out_codes = static_cast<uint8_t *>(x.out_codes);
  p.out_scales = static_cast<uint8_t *>(x.out_scales);
  p.status = x.status;
  p.test_timeout = (x.flags & PA_FLAG_TEST_WAIT_TIMEOUT) ? 1 : 0;
  e = ensure_smem_attr(reinterpret_cast<const void *>(pa_drafter_attn_kernel), kDaSmem);
  if (e != cudaSuccess) return record_cuda_error(e);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.maxp, (unsigned)x.R);
  cfg.blockDim = dim3(kDaThreads);
  cfg.dynamicSmemBytes = kDaSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (x.prof_before && (e = cudaEventRecord(static_cast<cudaEvent_t>(x.prof_before), s)) != cudaSuccess)
    return record_cuda_error(e);
  e = cudaLaunchKernelEx(&cfg, pa_drafter_attn_kernel, tmQ, tmKV, p, pdl ? 1 : 0);
  if (e != cudaSuccess) return record_cuda_error(e);
  if (x.prof_after && (e = cudaEventRecord(static_cast<cudaEvent_t>(x.prof_after), s)) != cudaSuccess)
    return record_cuda_error(e);
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3((unsigned)M);
  mcfg.blockDim = dim3(kDaMergeThreads);
  mcfg.stream = s;
  mcfg.attrs = attr;
  mcfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&mcfg, pa_drafter_merge_kernel, p, pdl ? 1 : 0);
  return e == cudaSuccess ? PA_OK : record_cuda_error(e);
}
