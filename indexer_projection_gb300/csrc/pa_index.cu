// Indexer scores ("vllm.models.minimax_m3.amd.mono.kernels.pre_attn",
// emit_k1: after the step every CTA scores the requests' index keys against
// the step's index_q; build_pre_attn_kernel: index_scale_log2e(sm_scale) and
// the sparse pinned init / local blocks).  emit_index_scores' body is not
// printed; this computes the reading the oracle states:
//   row m = r * q_len + i of request r sits at position p = seq_len[r] - q_len + i;
//   its page-128 blocks are b < nb = p / 128 + 1, the pinned ones (b < init
//   or b >= nb - local) get -inf, and key j (block j / 128, index slot
//   block_table[r][j / 128] * 128 + j % 128 of the FP8 index cache) gets
//     index_scale * sum_d bf16(index_q[m][d]) * e4m3(key_j[d])   (j <= p)
//   or -inf (j > p); columns from nb * 128 on are not written.
//
// The work is a skinny contraction (128 keys x 128 dims by up to 16 query
// rows per block) over a key stream that HBM bounds.  Up to 512 requests, a
// persistent grid (three CTAs an SM) walks the list of (request, block)
// items in even contiguous slices, a producer warp keeping four key blocks
// in flight a CTA (pa_index_scores_persist_kernel); beyond that, a CTA takes
// up to four blocks of one request (strided, for balance across the
// request's blocks; pa_index_scores_kernel).  Each block's 16 KB of keys
// arrives by one TMA copy (128-byte swizzle, so the fragment loads below hit
// distinct banks), and 8 warps take 16 keys each: ldmatrix reads a warp's 16 keys x 32 dims of E4M3 as four 8 x 8
// b16 tiles (2 E4M3 per b16), each thread converts its 4-code pieces to
// bf16 (exact: every E4M3 value is a bf16 value) and feeds
// mma.sync m16n8k16 bf16 with the query rows as B.  A thread's 4 codes of a
// piece are dims 4t .. 4t + 3 of the piece, so the MMA's k order is a
// permutation of the dims, applied to the query fragments alike (a dot
// product does not depend on the order of its terms).  f32 accumulation.
//
// The index_q rows are read after waiting on the previous kernel
// (programmatic dependent launch), so the scorer can follow pre_attn_run on
// the same stream.  Every wait is bounded (PA_DEV_WAIT_TIMEOUT); block ids
// outside the cache and rows the block table cannot hold are skipped and
// flagged (PA_DEV_SLOT_RANGE).
#include <cstdint>

#include "../../include/pre_attn.h"
#include "pa_device.cuh"
#include "pa_launch.h"
#include "pa_tma.h"

namespace pa {

constexpr int kIdxThreads = 256;       // 8 warps x 16 keys = one 128-key block
constexpr int kIdxBlocksPerCta = 4;    // blocks of one request a CTA takes
constexpr int kKeyBlockBytes = 128 * kHeadDim;  // 16 KB
constexpr int kIdxMaxRows = 16;        // q_len limit (two n8 tiles)
constexpr int kIdxSmem = kIdxBlocksPerCta * kKeyBlockBytes + 1024;  // + alignment slack

struct IndexParams {
  const __nv_bfloat16 *iq;  // row m at iq + m * iq_stride + head * 128
  int64_t iq_stride;
  int head;
  const uint8_t *index_cache;
  int64_t num_index_slots;
  const int32_t *block_table;
  const int32_t *seq_lens;
  int R, q_len, bt_width, init_blocks, local_blocks;
  float index_scale;
  float *scores;
  int64_t score_stride;
  uint32_t *status;
  uint64_t lim;      // bound of every wait (ns)
  int test_timeout;  // testing: the score warps also wait on a barrier nothing arrives on
};

__device__ __forceinline__ void tma_rows(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// 4 E4M3 codes (byte k = dim k of the piece) -> two bf16 pairs: .x holds
// codes 0, 1 (code 0 in the low half), .y codes 2, 3.  E4M3 -> f16 is exact
// (cvt), f16 -> f32 -> bf16 is exact for every E4M3 value.
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w) {
  uint32_t h[2];
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[0]) : "h"((uint16_t)(w & 0xffffu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[1]) : "h"((uint16_t)(w >> 16)));
  uint32_t o[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float lo = __half2float(__ushort_as_half((uint16_t)(h[i] & 0xffffu)));
    const float hi = __half2float(__ushort_as_half((uint16_t)(h[i] >> 16)));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[i]) : "f"(hi), "f"(lo));
  }
  return make_uint2(o[0], o[1]);
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The f16 variant.  Every E4M3 code is an f16 value, so a key converts in one
// instruction a pair (cvt.rn.f16x2.e4m3x2) instead of four through f32 and
// bf16; a bf16 query value is an f16 value when it is 0 or 2^-17 <= |x| <
// 2^15 (its 8 significant bits then sit on the f16 grid), so where every
// query value of a warp's fragments is, the products and the f32 sums are
// those of the bf16 MMA.  Otherwise (a value outside that range) the warp
// keeps the bf16 path for the request.
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint2 e4m3x4_to_f16x4(uint32_t w) {
  uint32_t h[2];
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[0]) : "h"((uint16_t)(w & 0xffffu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[1]) : "h"((uint16_t)(w >> 16)));
  return make_uint2(h[0], h[1]);
}
__device__ __forceinline__ bool bf16_on_f16_grid(uint32_t b) {  // b: 16 bf16 bits
  const uint32_t e = (b >> 7) & 0xffu;
  return (b & 0x7fffu) == 0 || (e >= 127 - 17 && e < 127 + 15);
}
// The query fragments of a thread as f16 pairs, in place, when every value
// of the warp's fragments is on the f16 grid; returns whether they are.
template <int NT>
__device__ __forceinline__ bool q_to_f16(uint2 (&qf)[NT][8]) {
  bool ok = true;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int pc = 0; pc < 8; ++pc) {
      const uint32_t w[2] = {qf[nt][pc].x, qf[nt][pc].y};
#pragma unroll
      for (int u = 0; u < 2; ++u) ok &= bf16_on_f16_grid(w[u] & 0xffffu) & bf16_on_f16_grid(w[u] >> 16);
    }
  ok = __all_sync(0xffffffffu, ok);
  if (ok) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) {
        uint32_t w[2] = {qf[nt][pc].x, qf[nt][pc].y};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float lo = bf16_to_f32(w[u] & 0xffffu), hi = bf16_to_f32(w[u] >> 16);
          asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w[u]) : "f"(hi), "f"(lo));
        }
        qf[nt][pc] = make_uint2(w[0], w[1]);
      }
  }
  return ok;
}

// Whether row (position p, nb = p / 128 + 1) takes a score in block b, and
// whether block b is one of its blocks at all.
__device__ __forceinline__ bool row_has_block(int64_t p, int b) { return p >= 0 && b <= p / 128; }
__device__ __forceinline__ bool row_scores_block(int64_t p, int b, int init, int local) {
  if (!row_has_block(p, b)) return false;
  const int64_t nb = p / 128 + 1;
  return b >= init && b < nb - local;
}

template <int NT>  // n8 tiles of query rows: q_len <= 8 * NT
__global__ void __launch_bounds__(kIdxThreads) pa_index_scores_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                      IndexParams a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ __align__(8) uint64_t full[kIdxBlocksPerCta];
  __shared__ __align__(8) uint64_t never;  // testing: nothing arrives on it
  __shared__ int blk_s[kIdxBlocksPerCta];  // block id, -1: not loaded
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int r = blockIdx.y;
  pdl_wait();  // the index_q rows (and new keys) come from the previous kernel
  const int seq = __ldg(a.seq_lens + r);
  const int64_t p_last = (int64_t)seq - 1;
  if (p_last < 0) return;
  const int nb_max = (int)(p_last / 128) + 1;
  const int64_t p_first = (int64_t)seq - a.q_len;
  if (tid == 0) {
    if (p_first < 0 || nb_max > a.bt_width) set_status(a.status, kDevSlotRange);
    for (int k = 0; k < kIdxBlocksPerCta; ++k) {
      mbar_init(&full[k], 1);
      blk_s[k] = -1;
    }
    mbar_init(&never, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (p_first < 0 || nb_max > a.bt_width) return;
  // this CTA's blocks: b = blockIdx.x + gridDim.x * k
  if (tid == 0) {
    for (int k = 0; k < kIdxBlocksPerCta; ++k) {
      const int b = blockIdx.x + gridDim.x * k;
      if (b >= nb_max) break;
      bool need = false;  // some row of the request scores this block
      for (int i = 0; i < a.q_len; ++i) need |= row_scores_block(p_first + i, b, a.init_blocks, a.local_blocks);
      if (!need) continue;
      const int64_t blk = __ldg(a.block_table + (int64_t)r * a.bt_width + b);
      if (blk < 0 || (blk + 1) * 128 > a.num_index_slots) {
        set_status(a.status, kDevSlotRange);
        continue;
      }
      blk_s[k] = (int)blk;
      mbar_expect_tx(&full[k], kKeyBlockBytes);
      tma_rows(smem_u32(smem + k * kKeyBlockBytes), &tmK, 0, (int)(blk * 128), &full[k]);
    }
  }
  // the query rows as B fragments: n8 tile nt, column g = row 8 nt + g; piece
  // (L, half) holds dims 32 L + 16 half + 4 t .. + 3 of that row (4 bf16)
  uint2 qf[NT][8];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int i = 8 * nt + g;
    const __nv_bfloat16 *row = a.iq + ((int64_t)r * a.q_len + i) * a.iq_stride + a.head * kHeadDim;
#pragma unroll
    for (int pc = 0; pc < 8; ++pc)
      qf[nt][pc] = i < a.q_len ? *reinterpret_cast<const uint2 *>(row + 16 * pc + 4 * t) : make_uint2(0u, 0u);
  }
  const bool qh = q_to_f16<NT>(qf);
  // rows of this thread's accumulator columns: 2t, 2t + 1 of each n8 tile
  int64_t prow[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = 8 * nt + 2 * t + e;
      prow[nt][e] = i < a.q_len ? p_first + i : -1;
    }
  __syncthreads();  // blk_s
  for (int k = 0; k < kIdxBlocksPerCta; ++k) {
    const int b = blockIdx.x + gridDim.x * k;
    if (b >= nb_max) break;
    const bool loaded = blk_s[k] >= 0;
    float c[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) c[nt][e] = 0.f;
    bool ok = true;
    if (loaded) {
      ok = mbar_wait(&full[k], 0, a.status, a.lim);
      if (ok && a.test_timeout) ok = mbar_wait(&never, 0, a.status, a.lim);
      if (ok) {
        const uint32_t base = smem_u32(smem + k * kKeyBlockBytes);
        // ldmatrix: thread l gives row (l & 7) of tile (l >> 3): key 16 warp +
        // 8 (tile & 1) + (l & 7), 16-byte chunk 2 L + (tile >> 1), swizzled
        const int key = 16 * warp + 8 * ((lane >> 3) & 1) + (lane & 7);
        const uint32_t rowaddr = base + key * 128;
#pragma unroll
        for (int L = 0; L < 4; ++L) {
          uint32_t m[4];
          const int chunk = 2 * L + (lane >> 4);
          ldmatrix_x4(rowaddr + ((chunk ^ (key & 7)) << 4), m);
          if (qh) {
            const uint2 k0 = e4m3x4_to_f16x4(m[0]), k1 = e4m3x4_to_f16x4(m[1]);  // keys g, g + 8: half 0
            const uint2 k2 = e4m3x4_to_f16x4(m[2]), k3 = e4m3x4_to_f16x4(m[3]);  // half 1
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_f16_16816(c[nt], k0.x, k1.x, k0.y, k1.y, qf[nt][2 * L].x, qf[nt][2 * L].y);
              mma_f16_16816(c[nt], k2.x, k3.x, k2.y, k3.y, qf[nt][2 * L + 1].x, qf[nt][2 * L + 1].y);
            }
          } else {
            const uint2 k0 = e4m3x4_to_bf16x4(m[0]), k1 = e4m3x4_to_bf16x4(m[1]);
            const uint2 k2 = e4m3x4_to_bf16x4(m[2]), k3 = e4m3x4_to_bf16x4(m[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_bf16_16816(c[nt], k0.x, k1.x, k0.y, k1.y, qf[nt][2 * L].x, qf[nt][2 * L].y);
              mma_bf16_16816(c[nt], k2.x, k3.x, k2.y, k3.y, qf[nt][2 * L + 1].x, qf[nt][2 * L + 1].y);
            }
          }
        }
      }
    }
    // scores of keys j0 = 128 b + 16 warp + g and j0 + 8 for this thread's rows
    const int64_t j0 = (int64_t)b * 128 + 16 * warp + g;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int64_t p = prow[nt][e];
        if (!row_has_block(p, b)) continue;
        const bool scored = row_scores_block(p, b, a.init_blocks, a.local_blocks);
        if (scored && !(loaded && ok)) continue;  // a key block that could not be read: left unwritten
        float *out = a.scores + ((int64_t)r * a.q_len + 8 * nt + 2 * t + e) * a.score_stride;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t j = j0 + 8 * h;
          out[j] = (scored && j <= p) ? c[nt][2 * h + e] * a.index_scale : -INFINITY;
        }
      }
  }
}

// ------------------------------------------------------ persistent variant
// Up to kIxPersistMaxR requests: a grid of three CTAs an SM walks the global
// list of (request, block) items, request by request, each CTA an even
// contiguous slice of it, so the key stream does not stop at CTA
// boundaries.  A producer warp keeps kIxStages key blocks in flight through
// a TMA ring; the eight compute warps score each block as the kernel above
// (the same fragments, the same masks and stores) and reload the query
// fragments only when the request changes.  Every CTA derives the item list
// itself: each request's block count from seq_lens, then a prefix sum.
constexpr int kIxStages = 4;
constexpr int kIxComputeWarps = 8;
constexpr int kIxPersistThreads = 32 * (kIxComputeWarps + 1);
constexpr int kIxPersistMaxR = 512;
constexpr int kIxPersistSmem = kIxStages * kKeyBlockBytes + 1024;  // + alignment slack

// Blocks of request r's score rows; 0 for a request without rows, and 0 with
// *bad set for one shorter than q_len or longer than its block table.
__device__ __forceinline__ int request_blocks(const IndexParams &a, int r, bool *bad) {
  const int seq = __ldg(a.seq_lens + r);
  if (seq < 1) return 0;
  const int nb = (seq - 1) / 128 + 1;
  if (seq < a.q_len || nb > a.bt_width) {
    *bad = true;
    return 0;
  }
  return nb;
}
// Whether some row of request r (rows at positions p_first .. p_first + q_len - 1) scores block b.
__device__ __forceinline__ bool block_needed(const IndexParams &a, int64_t p_first, int b) {
  for (int i = 0; i < a.q_len; ++i)
    if (row_scores_block(p_first + i, b, a.init_blocks, a.local_blocks)) return true;
  return false;
}
// Block id of (r, b) if it holds keys inside the cache, else -1.
__device__ __forceinline__ int64_t key_block(const IndexParams &a, int r, int b) {
  const int64_t blk = __ldg(a.block_table + (int64_t)r * a.bt_width + b);
  return (blk < 0 || (blk + 1) * 128 > a.num_index_slots) ? -1 : blk;
}

template <int NT>
__global__ void __launch_bounds__(kIxPersistThreads) pa_index_scores_persist_kernel(
    const __grid_constant__ CUtensorMap tmK, IndexParams a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ __align__(8) uint64_t full[kIxStages], empty[kIxStages];
  __shared__ __align__(8) uint64_t never;  // testing: nothing arrives on it
  __shared__ int offs[kIxPersistMaxR + 1];  // items before request r
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  pdl_wait();  // the index_q rows (and new keys) come from the previous kernel
  // each request's block count, then the prefix sum (warp 0: 16 requests a lane)
  if (warp == 0) {
    constexpr int kPer = (kIxPersistMaxR + 31) / 32;
    int cnt[kPer], sum = 0;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int r = lane * kPer + k;
      cnt[k] = r < a.R ? request_blocks(a, r, &bad) : 0;
      sum += cnt[k];
    }
    if (blockIdx.x == 0 && __any_sync(0xffffffffu, bad) && lane == 0) set_status(a.status, kDevSlotRange);
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int r = lane * kPer + k;
      if (r <= a.R) offs[r] = run;
      run += cnt[k];
    }
    if (lane == 31 && 32 * kPer == a.R) offs[a.R] = incl;
  }
  if (tid == 0) {
    for (int s = 0; s < kIxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kIxComputeWarps);
    }
    mbar_init(&never, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t total = offs[a.R];
  const int64_t lo = total * blockIdx.x / gridDim.x, hi = total * (blockIdx.x + 1) / gridDim.x;
  if (lo >= hi) return;
  int r0 = 0;  // the request of item lo: the last r with offs[r] <= lo
  for (int step = kIxPersistMaxR; step > 0; step >>= 1)
    if (r0 + step < a.R && offs[r0 + step] <= lo) r0 += step;
  // Items are resolved 32 at a time, one a lane (its request, block, whether
  // its keys are loaded and from which block), so the block-table reads of a
  // batch overlap instead of preceding each copy.
  struct Item {
    int r, b;
    int64_t blk;  // >= 0: its keys are loaded from this block
  };
  auto resolve = [&](int64_t idx, int r_from) {
    Item it{r_from, 0, -1};
    if (idx >= hi) return it;
    while (offs[it.r + 1] <= idx) ++it.r;
    it.b = (int)(idx - offs[it.r]);
    const int64_t pf = (int64_t)__ldg(a.seq_lens + it.r) - a.q_len;
    if (block_needed(a, pf, it.b)) {
      it.blk = key_block(a, it.r, it.b);
      if (it.blk < 0) it.blk = -2;  // needed but outside the cache: flagged, not loaded
    }
    return it;
  };
  if (warp == kIxComputeWarps) {
    // ------------------------------------------------------------ producer
    int j = 0, r = r0;
    bool ok = true;
    for (int64_t base = lo; base < hi && ok; base += 32) {
      const Item mine = resolve(base + lane, r);
      r = __shfl_sync(0xffffffffu, mine.r, 31);  // items are in request order
      for (int k = 0; k < 32 && base + k < hi; ++k) {
        const int64_t blk = __shfl_sync(0xffffffffu, mine.blk, k);
        if (blk == -2 && lane == 0) set_status(a.status, kDevSlotRange);
        if (blk < 0) continue;
        const int s = j % kIxStages;
        if (lane == 0) {
          if (!mbar_wait(&empty[s], ((uint32_t)(j / kIxStages) & 1) ^ 1, a.status, a.lim)) ok = false;
          else {
            mbar_expect_tx(&full[s], kKeyBlockBytes);
            tma_rows(smem_u32(smem + s * kKeyBlockBytes), &tmK, 0, (int)(blk * 128), &full[s]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++j;
      }
    }
    // the copies issued land before the CTA exits (they have, unless a wait ran out)
    if (lane == 0)
      for (int k = j - 1; k >= 0 && k >= j - kIxStages; --k)
        mbar_wait(&full[k % kIxStages], (uint32_t)(k / kIxStages) & 1, a.status, a.lim);
    return;
  }
  // ------------------------------------------------------------ compute
  int j = 0, cur = -1, r = r0;
  uint2 qf[NT][8];
  int64_t prow[NT][2];
  bool qh = false;  // the fragments hold f16 values
  for (int64_t base = lo; base < hi; base += 32) {
    const Item mine = resolve(base + lane, r);
    r = __shfl_sync(0xffffffffu, mine.r, 31);
    bool stop = false;
    for (int k = 0; k < 32 && base + k < hi; ++k) {
      const int ri = __shfl_sync(0xffffffffu, mine.r, k);
      const int b = __shfl_sync(0xffffffffu, mine.b, k);
      const bool loaded = __shfl_sync(0xffffffffu, mine.blk, k) >= 0;
      if (ri != cur) {  // the request's query fragments and row positions
        cur = ri;
        const int64_t p_first = (int64_t)__ldg(a.seq_lens + ri) - a.q_len;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int i = 8 * nt + g;
          const __nv_bfloat16 *row = a.iq + ((int64_t)ri * a.q_len + i) * a.iq_stride + a.head * kHeadDim;
#pragma unroll
          for (int pc = 0; pc < 8; ++pc)
            qf[nt][pc] = i < a.q_len ? *reinterpret_cast<const uint2 *>(row + 16 * pc + 4 * t) : make_uint2(0u, 0u);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int ii = 8 * nt + 2 * t + e;
            prow[nt][e] = ii < a.q_len ? p_first + ii : -1;
          }
        }
        qh = q_to_f16<NT>(qf);
      }
      float c[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[nt][e] = 0.f;
      if (loaded) {
        const int s = j % kIxStages;
        bool got = mbar_wait(&full[s], (uint32_t)(j / kIxStages) & 1, a.status, a.lim);
        if (got && a.test_timeout) got = mbar_wait(&never, 0, a.status, a.lim);
        if (__any_sync(0xffffffffu, !got)) {  // the warp gives up together
          stop = true;
          break;
        }
        const uint32_t sbase = smem_u32(smem + s * kKeyBlockBytes);
        const int key = 16 * warp + 8 * ((lane >> 3) & 1) + (lane & 7);
        const uint32_t rowaddr = sbase + key * 128;
#pragma unroll
        for (int L = 0; L < 4; ++L) {
          uint32_t m[4];
          const int chunk = 2 * L + (lane >> 4);
          ldmatrix_x4(rowaddr + ((chunk ^ (key & 7)) << 4), m);
          if (qh) {
            const uint2 k0 = e4m3x4_to_f16x4(m[0]), k1 = e4m3x4_to_f16x4(m[1]);
            const uint2 k2 = e4m3x4_to_f16x4(m[2]), k3 = e4m3x4_to_f16x4(m[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_f16_16816(c[nt], k0.x, k1.x, k0.y, k1.y, qf[nt][2 * L].x, qf[nt][2 * L].y);
              mma_f16_16816(c[nt], k2.x, k3.x, k2.y, k3.y, qf[nt][2 * L + 1].x, qf[nt][2 * L + 1].y);
            }
          } else {
            const uint2 k0 = e4m3x4_to_bf16x4(m[0]), k1 = e4m3x4_to_bf16x4(m[1]);
            const uint2 k2 = e4m3x4_to_bf16x4(m[2]), k3 = e4m3x4_to_bf16x4(m[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_bf16_16816(c[nt], k0.x, k1.x, k0.y, k1.y, qf[nt][2 * L].x, qf[nt][2 * L].y);
              mma_bf16_16816(c[nt], k2.x, k3.x, k2.y, k3.y, qf[nt][2 * L + 1].x, qf[nt][2 * L + 1].y);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        ++j;
      }
      // scores of keys 128 b + 16 warp + g and + 8 for this thread's rows
      const int64_t j0 = (int64_t)b * 128 + 16 * warp + g;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int64_t p = prow[nt][e];
          if (!row_has_block(p, b)) continue;
          const bool scored = row_scores_block(p, b, a.init_blocks, a.local_blocks);
          if (scored && !loaded) continue;  // a key block outside the cache: left unwritten
          float *out = a.scores + ((int64_t)ri * a.q_len + 8 * nt + 2 * t + e) * a.score_stride;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int64_t jj = j0 + 8 * h;
            out[jj] = (scored && jj <= p) ? c[nt][2 * h + e] * a.index_scale : -INFINITY;
          }
        }
    }
    if (stop) break;
  }
}


cudaError_t launch_index_scores(const IndexParams &a, cudaStream_t stream) {
  CUtensorMap tmK;
  if (!map_rows_sw128(&tmK, a.index_cache, (uint64_t)a.num_index_slots, kHeadDim, kHeadDim, 128))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int sms = current_device_sms();
  if (a.R <= kIxPersistMaxR && sms > 0) {
    auto kern = a.q_len <= 8 ? pa_index_scores_persist_kernel<1> : pa_index_scores_persist_kernel<2>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), kIxPersistSmem);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(3 * sms);
    cfg.blockDim = dim3(kIxPersistThreads);
    cfg.dynamicSmemBytes = kIxPersistSmem;
    return cudaLaunchKernelEx(&cfg, kern, tmK, a);
  }
  auto kern = a.q_len <= 8 ? pa_index_scores_kernel<1> : pa_index_scores_kernel<2>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), kIdxSmem);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((a.bt_width + kIdxBlocksPerCta - 1) / kIdxBlocksPerCta, a.R);
  cfg.blockDim = dim3(kIdxThreads);
  cfg.dynamicSmemBytes = kIdxSmem;
  return cudaLaunchKernelEx(&cfg, kern, tmK, a);
}

}  // namespace pa

extern "C" float pre_attn_index_scale_log2e(float sm_scale) {
  return (float)((double)sm_scale * 1.4426950408889634);  // log2(e)
}

extern "C" int pre_attn_index_scores(const pa_index_args *in, void *stream) {
  if (!in) return PA_ERR_NULL;
  const pa_index_args &x = *in;
  if (!x.iq || !x.index_cache || !x.block_table || !x.seq_lens || !x.scores || !x.status) return PA_ERR_NULL;
  if (x.R < 0 || x.R > 65535 || x.q_len < 1 || x.q_len > pa::kIdxMaxRows || x.bt_width < 1 || x.head < 0)
    return PA_ERR_SHAPE;
  if (x.init_blocks < 0 || x.local_blocks < 0 || !(x.index_scale == x.index_scale)) return PA_ERR_CONFIG;
  if (x.flags & ~(uint32_t)PA_FLAG_TEST_WAIT_TIMEOUT) return PA_ERR_CONFIG;
  if (x.num_index_slots < 128 || x.num_index_slots % 128) return PA_ERR_SHAPE;
  if (x.iq_stride < (int64_t)(x.head + 1) * pa::kHeadDim || x.score_stride < (int64_t)x.bt_width * 128)
    return PA_ERR_SHAPE;
  const uintptr_t u16 = 15;
  if ((reinterpret_cast<uintptr_t>(x.index_cache) & u16) || (reinterpret_cast<uintptr_t>(x.iq) & 7) ||
      (x.iq_stride % 4) || (reinterpret_cast<uintptr_t>(x.scores) & 3) ||
      (reinterpret_cast<uintptr_t>(x.block_table) & 3) || (reinterpret_cast<uintptr_t>(x.seq_lens) & 3) ||
      (reinterpret_cast<uintptr_t>(x.status) & 3))
    return PA_ERR_ALIGN;
  if (x.R == 0) return PA_OK;
  pa::IndexParams a;
  a.iq = static_cast<const __nv_bfloat16 *>(x.iq);
  a.iq_stride = x.iq_stride;
  a.head = x.head;
  a.index_cache = static_cast<const uint8_t *>(x.index_cache);
  a.num_index_slots = x.num_index_slots;
  a.block_table = x.block_table;
  a.seq_lens = x.seq_lens;
  a.R = x.R;
  a.q_len = x.q_len;
  a.bt_width = x.bt_width;
  a.init_blocks = x.init_blocks;
  a.local_blocks = x.local_blocks;
  a.index_scale = x.index_scale;
  a.scores = x.scores;
  a.score_stride = x.score_stride;
  a.status = x.status;
  a.test_timeout = (x.flags & PA_FLAG_TEST_WAIT_TIMEOUT) ? 1 : 0;
  a.lim = a.test_timeout ? pa::kTestWaitNs : pa::kWaitNs;
  const cudaError_t e = pa::launch_index_scores(a, (cudaStream_t)stream);
  return e == cudaSuccess ? PA_OK : pa::record_cuda_error(e);
}
