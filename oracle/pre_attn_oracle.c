/*
 * Test infrastructure, not product code.
 *
 * A plain, slow, single-threaded CPU oracle for the MiniMax-M3 sparse-layer
 * pre-attention step (residual add -> Gemma RMSNorm -> FP8 activation quant ->
 * fused [q | k | v | index_q | index_k] projection -> per-head Gemma RMSNorm +
 * partial NeoX RoPE -> q / index_q outputs and FP8 or NVFP4 paged-cache
 * insertion).  Only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code with the CUDA path.
 *
 * Citations name the page and the symbol / section they restate:
 *   [K1]  "vllm.models.minimax_m3.amd.mono.kernels.pre_attn" (K1 mono_pre):
 *         module summary, emit_pre_attn (norm_quant, GEMV tasks, head tasks),
 *         head_norm_rope, head_rope_inputs, page16_of.
 *   [EPI] "vllm.models.minimax_m3.nvidia.ops.qkv_index_fused_epilogue":
 *         module summary, QkvIndexFusedEpilogueKernel (N layout, epilogue
 *         roles), prepare_SF (F8_128x4 scale layout), _nvfp4_cache_views,
 *         _nvfp4_quant32, _rms_norm, _rope64,
 *         minimax_m3_qkv_index_fused_epilogue (argument contract).
 *   [DA]  "vllm.models.minimax_m3.amd.mono.drafter.attention" (the DSpark
 *         drafter's attention): module summary, qkv_rows, window, kv_load,
 *         block_math, block_acc, store_partial, merge_task.
 *
 * Precision: where the pages fix f32 (the residual sum, the per-token and
 * per-group quantiser arithmetic) the oracle does the same f32 operation;
 * everything else (sums of squares, rsqrt, the projection's dot products,
 * the head norm and RoPE) is computed in double and rounded to f32 once,
 * at the point where the pages hold an f32 value.  Every integer decision
 * (an FP8 / FP4 code, a scale byte) is taken on that f32 value.
 *
 * Readings where the pages are silent are listed at each function and
 * collected in the design notes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_OK 0
#define ORA_ERR_ARG (-1)
#define ORA_ERR_POS (-2)
#define ORA_ERR_SLOT (-3)

#define HEAD_DIM 128
#define ROT_DIM 64
#define HALF_ROT 32
#define FP8_MAX 448.0f

/* ------------------------------------------------------------------ codecs */

/* bf16: the top 16 bits of an IEEE binary32; round-to-nearest-even. */
float ora_bf16_decode(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

uint16_t ora_bf16_encode(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) /* inf / nan: keep, quiet the nan */
    return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
  uint32_t keep = u >> 16, rest = u & 0xffffu;
  if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
  return (uint16_t)keep;
}

float ora_bf16_round(float f) { return ora_bf16_decode(ora_bf16_encode(f)); }

/* OCP FP8 E4M3 ("fn": no infinities, S.1111.111 is NaN): bias 7, three
 * mantissa bits, largest finite 448, subnormals m * 2^-9. */
static double e4m3_magnitude(int c) { /* c in 0..126 */
  int e = (c >> 3) & 15, m = c & 7;
  if (e == 0) return ldexp((double)m, -9);
  return ldexp(8.0 + m, e - 10); /* (1 + m/8) * 2^(e-7) */
}

float ora_e4m3_decode(uint8_t code) {
  int mag = code & 0x7f;
  if (mag == 0x7f) return NAN;
  double v = e4m3_magnitude(mag);
  return (float)((code & 0x80) ? -v : v);
}

/* Nearest E4M3 value, ties to the even code, magnitudes above 448 clamp to
 * 448 (satfinite); NaN stays NaN.  Brute force over the 127 magnitudes. */
uint8_t ora_e4m3_encode(float x) {
  if (isnan(x)) return 0x7f;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7e;
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c <= 126; ++c) {
    double d = fabs(e4m3_magnitude(c) - a);
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  return (uint8_t)(sign | best);
}

/* FP4 E2M1: magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}, sign in bit 3. */
static const double e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

float ora_e2m1_decode(uint8_t nib) {
  double v = e2m1_mag[nib & 7];
  return (float)((nib & 8) ? -v : v);
}

/* Nearest E2M1 value, ties to the even code, clamped to +-6 (satfinite). */
uint8_t ora_e2m1_encode(float x) {
  uint8_t sign = signbit(x) ? 8 : 0;
  double a = fabs((double)x);
  if (isnan(x)) return 7; /* not produced by this path */
  if (a >= 6.0) return sign | 7;
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double d = fabs(e2m1_mag[c] - a);
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  return (uint8_t)(sign | best);
}

/* E8M0: an unsigned power-of-two exponent with bias 127; 0xff is NaN. */
double ora_e8m0_decode(uint8_t code) {
  if (code == 0xff) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* f32 product rounded toward zero ([EPI] _nvfp4_quant32: "rz" multiply).
 * The double product of two floats is exact, so truncating it is exact. */
static float mul_rz(float a, float b) {
  double p = (double)a * (double)b;
  float f = (float)p;
  if (fabs((double)f) > fabs(p)) f = nextafterf(f, 0.0f);
  return f;
}

/* ------------------------------------------------------- quantiser rules */

/* Per-token FP8 scale ([K1] norm_quant; head tasks for K / V):
 * amax / 448 as an f32 divide, or 1 when amax == 0. */
float ora_fp8_scale(float amax) { return amax == 0.0f ? 1.0f : amax / FP8_MAX; }

/* MXFP8 block exponent.  Reading (the pages receive MXFP8 pre-quantised and
 * print no rule): the smallest power of two 2^e with 448 * 2^e >= amax, i.e.
 * the per-block analogue of "scale = amax / 448", so no element clips;
 * e = 0 for an all-zero block; clamped to E8M0's [-127, 127]. */
int ora_mx_exponent(float amax) {
  if (!(amax > 0.0f)) return 0;
  int e = -127;
  while (e < 127 && ldexp(448.0, e) < (double)amax) ++e;
  return e;
}

/* NVFP4 quantiser of one 16-element group ([EPI] _nvfp4_quant32): the scale
 * byte is E4M3(max(gmax * (1/6) [* 1/global], 2^-9)); each element becomes
 * E2M1(RZ(v * (1/sf) [* 1/global])) with round-to-nearest-even on the E2M1
 * grid; a zero magnitude keeps no sign.  has_gs = 0 is the unit-scale form
 * (index_k).  Nibbles are returned one per byte. */
void ora_nvfp4_group16(const float *v, int has_gs, float gs_inv, uint8_t *nib,
                       uint8_t *sf_code) {
  float gmax = 0.0f;
  for (int i = 0; i < 16; ++i) gmax = fmaxf(gmax, fabsf(v[i]));
  float a = gmax * (float)(1.0 / 6.0);
  if (has_gs) a = a * gs_inv;
  a = fmaxf(a, 0x1p-9f);
  uint8_t c = ora_e4m3_encode(a);
  float sf = ora_e4m3_decode(c);
  float r = 1.0f / sf;
  if (has_gs) r = r * gs_inv;
  for (int i = 0; i < 16; ++i) {
    uint8_t n = ora_e2m1_encode(mul_rz(v[i], r));
    if ((n & 7) == 0) n = 0;
    nib[i] = n;
  }
  *sf_code = c;
}

/* ----------------------------------------------------------- the config */

typedef struct {
  int hidden;         /* H (the projection's K), a multiple of 128 */
  int n_q, n_kv, n_iq, n_ik; /* head counts; n_ik is 1 on the pages */
  int weight_fmt;     /* 0: per-channel FP8 (ptpc), 1: MXFP8 block-32 */
  int cache_fmt;      /* 0: FP8 per-token-scale caches, 1: NVFP4 caches */
  int block_size;     /* page size in tokens (16 for the FP8 layout) */
  int kv_page_stride; /* FP8 page16_of: page-16 blocks per 128-token block */
  int static_kv_scale;/* FP8 caches: K / V scales fixed at 1 */
  float eps;
} ora_config;

typedef struct {
  /* FP8 layout ([K1] head tasks): per page16 and KV head, 2048 B of K in the
   * page-16 "SHUFFLE" order, 2048 B of V transposed, one f32 scale per token;
   * index cache: 128 e4m3 per index slot. */
  uint8_t *k_cache, *v_cache;
  float *k_scale, *v_scale;
  uint8_t *index_cache;
  int64_t num_pages16;      /* page16 count of k/v caches and scale arrays */
  int64_t num_index_slots;  /* rows of the FP8 index cache */
  /* NVFP4 layout ([EPI] _nvfp4_cache_views): pages of 2*n_kv (KV) or 1
   * (index) slots of block_size tokens x 72 B. */
  uint8_t *kv_cache;
  int64_t kv_pages, kv_page_bytes;
  uint8_t *idx_cache;
  int64_t idx_pages, idx_page_bytes;
  float k_global, v_global; /* NVFP4 dequantisation (global) scales */
} ora_caches;

typedef struct {
  uint16_t *residual; /* [M, H] bf16 (may be NULL) */
  uint16_t *q_bf16;   /* [M, n_q*128] (NULL: not written) */
  uint8_t *q_fp8;     /* [M, n_q*128] e4m3 */
  uint16_t *iq_bf16;  /* [M, n_iq*128] */
  uint8_t *iq_fp8;    /* [M, n_iq*128] e4m3, unit scale */
  float q_fp8_scale;  /* dequantisation scale of q_fp8 */
} ora_outputs;

static int n_heads(const ora_config *c) { return c->n_q + 2 * c->n_kv + c->n_iq + c->n_ik; }

/* -------------------------------------------------- step 1-3: the prologue */

/* One token row ([K1] norm_quant): acc = ar + res in f32 (residual out is
 * bf16(acc)); Gemma RMSNorm n = acc * rsqrt(mean(acc^2) + eps) * (1 + gamma)
 * on the unrounded acc; then the activation quantiser:
 *   ptpc ([K1]): s = amax / 448 (1 if 0), xq = e4m3(n / s) with a true f32
 *        divide; *x_scale = s.
 *   MX (reading, see ora_mx_exponent): per 32-element block an E8M0
 *        exponent e, xq = e4m3(n * 2^-e); xsf[b] = e + 127. */
int ora_prologue_row(const ora_config *c, const uint16_t *ar, const uint16_t *res,
                     const uint16_t *g_in, uint16_t *residual, uint8_t *xq,
                     float *x_scale, uint8_t *xsf) {
  const int H = c->hidden;
  float *acc = (float *)malloc(sizeof(float) * H);
  float *n = (float *)malloc(sizeof(float) * H);
  if (!acc || !n) { free(acc); free(n); return ORA_ERR_ARG; }
  double ss = 0.0;
  for (int k = 0; k < H; ++k) {
    acc[k] = ora_bf16_decode(ar[k]) + ora_bf16_decode(res[k]); /* f32 add */
    if (residual) residual[k] = ora_bf16_encode(acc[k]);
    ss += (double)acc[k] * (double)acc[k];
  }
  double rstd = 1.0 / sqrt(ss / H + (double)c->eps);
  for (int k = 0; k < H; ++k)
    n[k] = (float)((double)acc[k] * rstd * (1.0 + (double)ora_bf16_decode(g_in[k])));
  if (c->weight_fmt == 0) {
    float amax = 0.0f;
    for (int k = 0; k < H; ++k) amax = fmaxf(amax, fabsf(n[k]));
    float s = ora_fp8_scale(amax);
    for (int k = 0; k < H; ++k) xq[k] = ora_e4m3_encode(n[k] / s);
    *x_scale = s;
  } else {
    for (int b = 0; b < H / 32; ++b) {
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(n[32 * b + i]));
      int e = ora_mx_exponent(amax);
      float inv = (float)ldexp(1.0, -e);
      for (int i = 0; i < 32; ++i) xq[32 * b + i] = ora_e4m3_encode(n[32 * b + i] * inv);
      xsf[b] = (uint8_t)(e + 127);
    }
  }
  free(acc);
  free(n);
  return ORA_OK;
}

/* ------------------------------------------------ step 4: the projection */

/* y[n] for one token over all N = n_heads * 128 output channels, never
 * rounded to bf16 (north-star "f32 accumulator"; [EPI] summary):
 *   ptpc ([K1] GEMV tasks): y = (sum_k xq_k * w_nk) * x_scale * w_scale[n]
 *   MX ([EPI]): y = sum_b 2^(ea_b + eb_nb) * sum_{k in block b} xq_k * w_nk
 * The inner sums are exact in double; y is rounded to f32 once.
 * w is [N, H] e4m3 row-major (K-major); w_scale is [N] f32 (ptpc);
 * wsf is [N, H/32] E8M0 row-major (MX). */
void ora_project_row(const ora_config *c, const uint8_t *xq, float x_scale,
                     const uint8_t *xsf, const uint8_t *w, const float *w_scale,
                     const uint8_t *wsf, float *y) {
  const int H = c->hidden, N = n_heads(c) * HEAD_DIM;
  double *xv = (double *)malloc(sizeof(double) * H);
  double lut[256];
  for (int i = 0; i < 256; ++i) lut[i] = (double)ora_e4m3_decode((uint8_t)i);
  for (int k = 0; k < H; ++k) xv[k] = lut[xq[k]];
  for (int nn = 0; nn < N; ++nn) {
    const uint8_t *wr = w + (size_t)nn * H;
    if (c->weight_fmt == 0) {
      double s = 0.0;
      for (int k = 0; k < H; ++k) s += xv[k] * lut[wr[k]];
      y[nn] = (float)(s * (double)x_scale * (double)w_scale[nn]);
    } else {
      double tot = 0.0;
      for (int b = 0; b < H / 32; ++b) {
        double s = 0.0;
        for (int i = 0; i < 32; ++i) s += xv[32 * b + i] * lut[wr[32 * b + i]];
        tot += s * ora_e8m0_decode(xsf[b]) * ora_e8m0_decode(wsf[(size_t)nn * (H / 32) + b]);
      }
      y[nn] = (float)tot;
    }
  }
  free(xv);
}

/* ------------------------------------- step 5: head Gemma RMSNorm + RoPE */

/* Gemma RMSNorm of one 128-dim head ([K1] head_norm_rope, [EPI] _rms_norm):
 * z = y * rsqrt(mean(y^2) + eps) * (1 + gamma), in double. */
void ora_head_rmsnorm(const float *y, const uint16_t *gamma, float eps, double *z) {
  double ss = 0.0;
  for (int i = 0; i < HEAD_DIM; ++i) ss += (double)y[i] * (double)y[i];
  double rr = 1.0 / sqrt(ss / HEAD_DIM + (double)eps);
  for (int i = 0; i < HEAD_DIM; ++i)
    z[i] = (double)y[i] * rr * (1.0 + (double)ora_bf16_decode(gamma[i]));
}

/* Partial NeoX RoPE over dims [0, 64) ([K1] head_norm_rope /
 * head_rope_inputs, [EPI] _rope64): for i < 32, x = z[i], w = z[i + 32],
 * c = cos_sin[pos][i], s = cos_sin[pos][32 + i] (bf16 table [max_pos, 64]);
 * z[i] = x c - w s, z[i + 32] = w c + x s.  Dims [64, 128) are untouched. */
void ora_rope_neox(double *z, const uint16_t *cs_row) {
  for (int i = 0; i < HALF_ROT; ++i) {
    double cc = ora_bf16_decode(cs_row[i]), sn = ora_bf16_decode(cs_row[HALF_ROT + i]);
    double x = z[i], w = z[i + HALF_ROT];
    z[i] = x * cc - w * sn;
    z[i + HALF_ROT] = w * cc + x * sn;
  }
}

/* ------------------------------------------- step 7: cache address maps */

/* [K1] page16_of: the page-16 id of a slot; kps = the host's K / V block
 * page stride in page-16 units per 128-token sparse block (8 = identity). */
int64_t ora_page16_of(int64_t slot, int kps) {
  if (kps == 128 / 16) return slot / 16;
  return (slot / 128) * kps + (slot % 128) / 16;
}

/* FP8 K "SHUFFLE" page ([K1] head tasks, K store): byte of dim d, token t. */
int64_t ora_fp8_k_offset(int64_t page16, int h, int n_kv, int t, int d) {
  return (page16 * n_kv + h) * 2048 + (d / 16) * 256 + t * 16 + d % 16;
}
/* FP8 V page ([K1] head tasks, V store): transposed, byte d * 16 + t. */
int64_t ora_fp8_v_offset(int64_t page16, int h, int n_kv, int t, int d) {
  return (page16 * n_kv + h) * 2048 + d * 16 + t;
}
/* f32 per-token K / V scale index ([K1]: b * PAGE16 + t, per KV head). */
int64_t ora_fp8_scale_index(int64_t page16, int h, int n_kv, int t) {
  return (page16 * n_kv + h) * 16 + t;
}

/* NVFP4 page ([EPI] _nvfp4_cache_views): slot s of a page holds bs tokens'
 * E2M1 data (64 B a token: [half][32 B]) then their 8 E4M3 scale bytes.
 * Reading: inside a data byte the even element is the low nibble. */
int64_t ora_nvfp4_data_offset(int bs, int slot_in_page, int t, int d) {
  int64_t slot_bytes = (int64_t)bs * 72;
  return slot_in_page * slot_bytes + (int64_t)t * 64 + (d / 64) * 32 + (d % 64) / 2;
}
/* Linear scale byte g (dims 16g..16g+15) of token t (K and index_k). */
int64_t ora_nvfp4_sf_linear_offset(int bs, int slot_in_page, int t, int g) {
  return slot_in_page * (int64_t)bs * 72 + (int64_t)bs * 64 + (int64_t)t * 8 + g;
}
/* V-swizzled scale byte g of token t: (t/4*4 + g/2) * 8 + g%2 * 4 + t%4. */
int64_t ora_nvfp4_sf_vswz_offset(int bs, int slot_in_page, int t, int g) {
  return slot_in_page * (int64_t)bs * 72 + (int64_t)bs * 64 +
         (int64_t)((t / 4) * 4 + g / 2) * 8 + (g % 2) * 4 + t % 4;
}

/* F8_128x4 scale-factor layout ([EPI] prepare_SF): the grid [R, Ksf] padded
 * to R % 128 == 0 and permuted as [R/128, Ksf/4, 32, 4, 4]; the [32, 4, 4]
 * atom indexes (row % 32, (row % 128) / 32, k-block % 4). */
int64_t ora_sf128x4_offset(int64_t r, int64_t kb, int64_t ksf) {
  return ((r / 128) * (ksf / 4) + kb / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4;
}

void ora_pack_sf128x4(const uint8_t *src, int64_t rows, int64_t ksf, uint8_t *dst, uint8_t pad) {
  int64_t rpad = (rows + 127) / 128 * 128;
  memset(dst, pad, (size_t)(rpad * ksf));
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t kb = 0; kb < ksf; ++kb) dst[ora_sf128x4_offset(r, kb, ksf)] = src[r * ksf + kb];
}

/* -------------------------------------------------- steps 5-7 per token */

typedef struct {
  const uint16_t *g_q, *g_k, *g_iq, *g_ik; /* [128] bf16 head gammas */
  const uint16_t *cos_sin;                 /* [max_pos, 64] bf16 */
  int64_t max_pos;
} ora_head_params;

static void fp8_cache_store(const ora_config *c, const ora_caches *cc, int kv_head, int is_v,
                            int64_t slot, const float *vals, int bf16_first) {
  int64_t p16 = ora_page16_of(slot, c->kv_page_stride);
  int t = (int)(slot % 16);
  float amax = 0.0f;
  for (int i = 0; i < HEAD_DIM; ++i) amax = fmaxf(amax, fabsf(vals[i]));
  float s = c->static_kv_scale ? 1.0f : ora_fp8_scale(amax);
  for (int d = 0; d < HEAD_DIM; ++d) {
    float v = bf16_first ? ora_bf16_round(vals[d]) : vals[d];
    uint8_t code = ora_e4m3_encode(v / s);
    if (is_v) cc->v_cache[ora_fp8_v_offset(p16, kv_head, c->n_kv, t, d)] = code;
    else cc->k_cache[ora_fp8_k_offset(p16, kv_head, c->n_kv, t, d)] = code;
  }
  int64_t si = ora_fp8_scale_index(p16, kv_head, c->n_kv, t);
  if (is_v) cc->v_scale[si] = s;
  else cc->k_scale[si] = s;
}

static void nvfp4_store(uint8_t *page, int bs, int slot_in_page, int t, const float *vals,
                        int has_gs, float gs_inv, int v_swizzle) {
  for (int g = 0; g < 8; ++g) {
    uint8_t nib[16], sf;
    ora_nvfp4_group16(vals + 16 * g, has_gs, gs_inv, nib, &sf);
    for (int i = 0; i < 16; i += 2) {
      int d = 16 * g + i;
      page[ora_nvfp4_data_offset(bs, slot_in_page, t, d)] = (uint8_t)(nib[i] | (nib[i + 1] << 4));
    }
    int64_t so = v_swizzle ? ora_nvfp4_sf_vswz_offset(bs, slot_in_page, t, g)
                           : ora_nvfp4_sf_linear_offset(bs, slot_in_page, t, g);
    page[so] = sf;
  }
}

/* The per-head epilogue of one token ([K1] head tasks, [EPI] kernel epilogue
 * roles).  Heads are [q x n_q | k x n_kv | v x n_kv | index_q x n_iq |
 * index_k x 1] ([EPI] QkvIndexFusedEpilogueKernel.__init__).
 *   q, index_q, k, index_k: Gemma RMSNorm + RoPE; v: the raw projection.
 *   q out: bf16(z) and / or e4m3(z * (1 / q_fp8_scale)) ([EPI] q branch).
 *   index_q out: bf16(z) ([K1]) and / or e4m3(z), unit scale ([EPI]).
 *   FP8 caches ([K1]): K codes e4m3(bf16(z) / ks), ks from amax(z);
 *     V codes e4m3(y / vs), vs from amax(y); index_k e4m3(bf16(z)).
 *   NVFP4 caches ([EPI]): K with 1/k_global, V with 1/v_global and the
 *     swizzled scale bytes, index_k at unit scale.
 * slot < 0 skips every store of that cache ([EPI] slot_mapping "-1 = skip"). */
int ora_heads_row(const ora_config *c, const ora_head_params *hp, const float *y, int64_t pos,
                  int64_t slot, int64_t islot, const ora_caches *cc, const ora_outputs *o,
                  int64_t m) {
  if (pos < 0 || pos >= hp->max_pos) return ORA_ERR_POS;
  const uint16_t *cs_row = hp->cos_sin + pos * ROT_DIM;
  const int k0 = c->n_q, v0 = k0 + c->n_kv, iq0 = v0 + c->n_kv, ik0 = iq0 + c->n_iq;
  const int nh = n_heads(c);
  const int bs = c->block_size;
  /* bounds of the slots, checked before anything is written */
  if (slot >= 0) {
    if (c->cache_fmt == 0) {
      if (ora_page16_of(slot, c->kv_page_stride) >= cc->num_pages16) return ORA_ERR_SLOT;
    } else if (slot / bs >= cc->kv_pages) return ORA_ERR_SLOT;
  }
  if (islot >= 0) {
    if (c->cache_fmt == 0) {
      if (islot >= cc->num_index_slots) return ORA_ERR_SLOT;
    } else if (islot / bs >= cc->idx_pages) return ORA_ERR_SLOT;
  }
  float zf[HEAD_DIM];
  double z[HEAD_DIM];
  for (int hh = 0; hh < nh; ++hh) {
    const float *yh = y + (size_t)hh * HEAD_DIM;
    const uint16_t *gamma = hh < k0 ? hp->g_q : hh < v0 ? hp->g_k : hh < iq0 ? NULL
                          : hh < ik0 ? hp->g_iq : hp->g_ik;
    if (hh >= v0 && hh < iq0) {
      for (int i = 0; i < HEAD_DIM; ++i) zf[i] = yh[i];
    } else {
      ora_head_rmsnorm(yh, gamma, c->eps, z);
      ora_rope_neox(z, cs_row);
      for (int i = 0; i < HEAD_DIM; ++i) zf[i] = (float)z[i];
    }
    if (hh < k0) { /* q */
      size_t base = (size_t)m * c->n_q * HEAD_DIM + (size_t)hh * HEAD_DIM;
      float inv = 1.0f / o->q_fp8_scale;
      for (int i = 0; i < HEAD_DIM; ++i) {
        if (o->q_bf16) o->q_bf16[base + i] = ora_bf16_encode(zf[i]);
        if (o->q_fp8) o->q_fp8[base + i] = ora_e4m3_encode(zf[i] * inv);
      }
    } else if (hh < v0) { /* k */
      int h = hh - k0;
      if (slot < 0) continue;
      if (c->cache_fmt == 0) {
        fp8_cache_store(c, cc, h, 0, slot, zf, 1);
      } else {
        uint8_t *page = cc->kv_cache + (slot / bs) * cc->kv_page_bytes;
        nvfp4_store(page, bs, 2 * h, (int)(slot % bs), zf, 1, 1.0f / cc->k_global, 0);
      }
    } else if (hh < iq0) { /* v */
      int h = hh - v0;
      if (slot < 0) continue;
      if (c->cache_fmt == 0) {
        fp8_cache_store(c, cc, h, 1, slot, zf, 0);
      } else {
        uint8_t *page = cc->kv_cache + (slot / bs) * cc->kv_page_bytes;
        nvfp4_store(page, bs, 2 * h + 1, (int)(slot % bs), zf, 1, 1.0f / cc->v_global, 1);
      }
    } else if (hh < ik0) { /* index_q */
      size_t base = (size_t)m * c->n_iq * HEAD_DIM + (size_t)(hh - iq0) * HEAD_DIM;
      for (int i = 0; i < HEAD_DIM; ++i) {
        if (o->iq_bf16) o->iq_bf16[base + i] = ora_bf16_encode(zf[i]);
        if (o->iq_fp8) o->iq_fp8[base + i] = ora_e4m3_encode(zf[i]);
      }
    } else { /* index_k */
      if (islot < 0) continue;
      if (c->cache_fmt == 0) {
        for (int d = 0; d < HEAD_DIM; ++d)
          cc->index_cache[islot * HEAD_DIM + d] = ora_e4m3_encode(ora_bf16_round(zf[d]));
      } else {
        uint8_t *page = cc->idx_cache + (islot / bs) * cc->idx_page_bytes;
        nvfp4_store(page, bs, 0, (int)(islot % bs), zf, 0, 1.0f, 0);
      }
    }
  }
  return ORA_OK;
}

/* ------------------------------------------------------ the whole step */

typedef struct {
  const uint16_t *ar, *res, *g_in; /* [M, H], [M, H], [H] bf16 */
  const uint8_t *w;                /* [N, H] e4m3 */
  const float *w_scale;            /* ptpc: [N] f32 */
  const uint8_t *wsf;              /* MX: [N, H/32] E8M0, row-major */
  const int64_t *positions, *slot_mapping, *index_slot_mapping; /* [M] */
} ora_inputs;

/* Rows [row0, row1) of the step; rows are independent, so callers may run
 * disjoint row ranges concurrently.  y_out (optional, [M, N] f32) receives
 * the projection, xq_out / xs_out (optional) the activation codes and
 * scales (ptpc: [M] f32 into xs_out; MX: [M, H/32] E8M0 codes into
 * xsf_out). */
int ora_pre_attn_rows(const ora_config *c, const ora_inputs *in, const ora_head_params *hp,
                      const ora_caches *cc, const ora_outputs *o, int64_t row0, int64_t row1,
                      float *y_out, uint8_t *xq_out, float *xs_out, uint8_t *xsf_out) {
  if (!c || !in || !hp || !cc || !o) return ORA_ERR_ARG;
  if (c->hidden <= 0 || c->hidden % 128 || c->n_kv <= 0 || c->n_ik != 1) return ORA_ERR_ARG;
  const int H = c->hidden, N = n_heads(c) * HEAD_DIM;
  uint8_t *xq = (uint8_t *)malloc(H);
  uint8_t *xsf = (uint8_t *)malloc(H / 32);
  float *y = (float *)malloc(sizeof(float) * N);
  int rc = ORA_OK;
  for (int64_t m = row0; m < row1 && rc == ORA_OK; ++m) {
    float xs = 1.0f;
    rc = ora_prologue_row(c, in->ar + m * H, in->res + m * H, in->g_in,
                          o->residual ? o->residual + m * H : NULL, xq, &xs, xsf);
    if (rc) break;
    ora_project_row(c, xq, xs, xsf, in->w, in->w_scale, in->wsf, y);
    int64_t slot = in->slot_mapping[m];
    int64_t islot = in->index_slot_mapping ? in->index_slot_mapping[m] : slot;
    rc = ora_heads_row(c, hp, y, in->positions[m], slot, islot, cc, o, m);
    if (y_out) memcpy(y_out + m * N, y, sizeof(float) * N);
    if (xq_out) memcpy(xq_out + m * H, xq, H);
    if (xs_out) xs_out[m] = xs;
    if (xsf_out && c->weight_fmt == 1) memcpy(xsf_out + m * (H / 32), xsf, H / 32);
  }
  free(xq);
  free(xsf);
  free(y);
  return rc;
}

/* ------------------------------------------------ the indexer scores */

/* index_scale_log2e(sm_scale) ([K1] build_pre_attn_kernel; the body is not
 * printed).  Reading: the attention scale times log2(e), so that
 * exp2(score) = exp(sm_scale * q.k), the scale an exp2-based softmax over the
 * scores takes. */
double ora_index_scale_log2e(double sm_scale) { return sm_scale * (1.0 / log(2.0)); }

/* The indexer scores of a step's rows ([K1] emit_k1: after the step, every
 * CTA scores the index keys of its requests against the step's index_q;
 * emit_index_scores' body is not printed, so this is a reading).
 * Rows: request r (r < R) has q_len consecutive rows m = r * q_len + i at
 * positions p = seq_lens[r] - q_len + i (the speculative verify rows).
 * Keys: key j of request r (j <= p: causal) sits in page-128 block
 * b = j / 128 at index slot block_table[r * bt_width + b] * 128 + j % 128 of
 * the FP8 index cache (E4M3, unit scale, 128 bytes a slot).  Row m's blocks
 * are b < nb = p / 128 + 1; the pinned ones (b < init_blocks, the first
 * blocks, or b >= nb - local_blocks, the local window) are attended anyway
 * and get no score.
 * Output, row m of scores (score_stride floats a row), columns j < nb * 128:
 *   index_scale * sum_d bf16(iq[m][d]) * e4m3(key_j[d])   j <= p, b not pinned
 *   -inf                                                    otherwise
 * The dot product is exact in double, rounded to f32 once after the scale.
 * Columns from nb * 128 on are not written.  iq row m starts at
 * iq + m * iq_stride (bf16).  Returns ORA_ERR_ARG for a row before position
 * 0 or beyond the block table, ORA_ERR_SLOT for a key outside the cache. */
int ora_index_scores(const uint16_t *iq, int64_t iq_stride, const uint8_t *index_cache,
                     int64_t num_index_slots, const int32_t *block_table, int bt_width,
                     const int32_t *seq_lens, int R, int q_len, int init_blocks, int local_blocks,
                     float index_scale, float *scores, int64_t score_stride) {
  double lut[256];
  for (int c = 0; c < 256; ++c) lut[c] = (double)ora_e4m3_decode((uint8_t)c);
  for (int r = 0; r < R; ++r) {
    for (int i = 0; i < q_len; ++i) {
      const int64_t m = (int64_t)r * q_len + i;
      const int64_t p = (int64_t)seq_lens[r] - q_len + i;
      if (p < 0) return ORA_ERR_ARG;
      const int64_t nb = p / 128 + 1;
      if (nb > bt_width || nb * 128 > score_stride) return ORA_ERR_ARG;
      double q[HEAD_DIM];
      for (int d = 0; d < HEAD_DIM; ++d) q[d] = ora_bf16_decode(iq[m * iq_stride + d]);
      for (int64_t b = 0; b < nb; ++b) {
        const int pinned = b < init_blocks || b >= nb - local_blocks;
        const int64_t blk = block_table[(int64_t)r * bt_width + b];
        for (int jj = 0; jj < 128; ++jj) {
          const int64_t j = b * 128 + jj;
          float out = -INFINITY;
          if (!pinned && j <= p) {
            const int64_t slot = blk * 128 + jj;
            if (blk < 0 || slot >= num_index_slots) return ORA_ERR_SLOT;
            const uint8_t *key = index_cache + slot * HEAD_DIM;
            double s = 0.0;
            for (int d = 0; d < HEAD_DIM; ++d) s += q[d] * lut[key[d]];
            out = (float)(s * (double)index_scale);
          }
          scores[m * score_stride + j] = out;
        }
      }
    }
  }
  return ORA_OK;
}


/* --------------------------------------------- the drafter's attention */

/* [DA] "vllm.models.minimax_m3.amd.mono.drafter.attention": the DSpark
 * drafter's attention over its own FP8 KV cache, one KV head of 128 dims, 16
 * query heads, up to 8 rows a request (7 on the page).  The drafter cache
 * holds page-128 blocks of 128 keys, 256 bytes a key: the key's 128 E4M3 K
 * bytes, then its 128 E4M3 V bytes (kv_load); q, K and V are unit-scale FP8
 * (module summary: "FP8 q"). */
#define DA_HEADS 16
#define DA_BLOCK 128
#define DA_KEY_BYTES 256

/* The drafter's q / k head norms, RoPE and FP8 (qkv_rows: "head norm, RoPE,
 * FP8"; its new K / V rows go to the cache).  Row m of qkv (qkv_stride bf16
 * values) holds 16 q heads, then k, then v, 128 each.  q and k take the
 * step's head norm (ora_head_rmsnorm with gamma qn / kn) and its partial NeoX
 * RoPE at positions[m] (a reading: the page names the steps, not their
 * form); v is taken as is.  q8 row (m * 16 + h) gets E4M3(f32(z)) of head h;
 * the key at slot slot_mapping[m] (slot < 0: none) gets E4M3(f32(k)) and
 * E4M3(v) at cache byte slot * 256 and slot * 256 + 128.  Returns
 * ORA_ERR_POS for a position outside [0, max_pos), ORA_ERR_SLOT for a slot
 * past the cache, before anything of that row is written. */
int ora_drafter_qkv(const uint16_t *qkv, int64_t qkv_stride, int64_t M, const uint16_t *qn,
                    const uint16_t *kn, float eps, const uint16_t *cos_sin, int64_t max_pos,
                    const int64_t *positions, const int64_t *slot_mapping, uint8_t *cache,
                    int64_t num_blocks, uint8_t *q8) {
  float y[HEAD_DIM];
  double z[HEAD_DIM];
  for (int64_t m = 0; m < M; ++m) {
    const int64_t pos = positions[m], slot = slot_mapping[m];
    if (pos < 0 || pos >= max_pos) return ORA_ERR_POS;
    if (slot >= num_blocks * DA_BLOCK) return ORA_ERR_SLOT;
    const uint16_t *cs = cos_sin + pos * ROT_DIM;
    for (int h = 0; h < DA_HEADS + 2; ++h) {
      const uint16_t *src = qkv + m * qkv_stride + (int64_t)h * HEAD_DIM;
      for (int d = 0; d < HEAD_DIM; ++d) y[d] = ora_bf16_decode(src[d]);
      if (h <= DA_HEADS) {
        ora_head_rmsnorm(y, h < DA_HEADS ? qn : kn, eps, z);
        ora_rope_neox(z, cs);
        for (int d = 0; d < HEAD_DIM; ++d) y[d] = (float)z[d];
      }
      uint8_t *dst = h < DA_HEADS ? q8 + (m * DA_HEADS + h) * HEAD_DIM
                   : slot < 0     ? NULL
                   : cache + slot * DA_KEY_BYTES + (h - DA_HEADS) * HEAD_DIM;
      if (!dst) continue;
      for (int d = 0; d < HEAD_DIM; ++d) dst[d] = ora_e4m3_encode(y[d]);
    }
  }
  return ORA_OK;
}

/* Request r's key window ([DA] window): rows r * q_len .. + q_len - 1 sit at
 * p0 + j with p0 = positions[r * q_len]; the keys lo .. hi with
 * lo = max(p0 - (window - 1), 0) and hi = min(seq_len - 1,
 * (lo / 128 + max_blocks) * 128 - 1), blocks lo / 128 .. hi / 128.  Key kp
 * counts for row j when lo <= kp <= hi and kp > p0 + j - window
 * (block_math's mask): the rows see each other's keys, non-causally. */
void ora_drafter_window(int64_t p0, int64_t seq, int window, int max_blocks, int64_t *lo,
                        int64_t *hi) {
  int64_t a = p0 - (window - 1);
  if (a < 0) a = 0;
  int64_t b = (a / DA_BLOCK + max_blocks) * DA_BLOCK - 1;
  if (seq - 1 < b) b = seq - 1;
  *lo = a;
  *hi = b;
}

/* The split-KV attention and its merge ([DA] module summary, block_acc,
 * block_math, store_partial, merge_task), for R requests of q_len rows.
 *   Partitions: the window's blocks, from lo / 128 on, in runs of
 *     part_blocks blocks (the page fixes the partition's math, not its
 *     length: a reading; the GPU path takes the same argument).  Each is an
 *     online softmax over its blocks in order: with C = sm_scale * log2(e)
 *     and m = -inf, l = 0, o = 0 to start, a block's valid scores s = q . k
 *     (raw units) give m' = max(m, max s), ms = (m' == -inf ? 0 : m'),
 *     alpha = exp2((m - ms) C), p = f32(exp2(s C - (ms C - 8))) (P x 256 at
 *     m'), l = l alpha + sum p, o = o alpha + sum E4M3(p) v.  l sums the
 *     unquantised p, o the E4M3 ones (block_acc).
 *   Merge, in partition order (merge_task): m* = max m_i, w_i =
 *     exp2((m_i - m*) C) (0 for a partition that saw no valid key), out =
 *     (sum w_i o_i) / (sum w_i l_i); a row with no valid key at all gives 0.
 *     out is rounded to bf16, then quantised to MXFP8 over the row's 16 * 128
 *     values: 32-value blocks, ora_mx_exponent's E8M0 exponent e, codes
 *     E4M3(x * 2^-e), scale byte e + 127.
 * Sums and products are exact or in double.  q8 row (m * 16 + h) holds head
 * h of row m; out_bf16 (optional) [R * q_len, 2048]; out_codes likewise
 * (bytes); out_scales [R * q_len, 64].  A request whose window is empty
 * (hi < lo) gets zero rows.  Returns ORA_ERR_ARG when a window block lies
 * past the block table, ORA_ERR_SLOT for a block id outside the cache. */
typedef struct {
  int R, q_len, bt_width;
  int window, max_blocks, part_blocks;
  double sm_scale;
} ora_dattn_cfg;

int ora_drafter_attention(const ora_dattn_cfg *c, const uint8_t *q8, const uint8_t *cache,
                          int64_t num_blocks, const int32_t *block_table, const int32_t *seq_lens,
                          const int64_t *positions, uint16_t *out_bf16, uint8_t *out_codes,
                          uint8_t *out_scales) {
  const double C = c->sm_scale / log(2.0);
  const int D = HEAD_DIM, W = DA_HEADS * HEAD_DIM;
  double lut[256];
  for (int i = 0; i < 256; ++i) lut[i] = (double)ora_e4m3_decode((uint8_t)i);
  const int maxp = (c->max_blocks + c->part_blocks - 1) / c->part_blocks + 1;
  double *pm = (double *)malloc(sizeof(double) * maxp);
  double *pl = (double *)malloc(sizeof(double) * maxp);
  double *po = (double *)malloc(sizeof(double) * maxp * D);
  float *row = (float *)malloc(sizeof(float) * W);
  if (!pm || !pl || !po || !row) {
    free(pm); free(pl); free(po); free(row);
    return ORA_ERR_ARG;
  }
  int rc = ORA_OK;
  for (int r = 0; r < c->R && rc == ORA_OK; ++r) {
    const int64_t p0 = positions[(int64_t)r * c->q_len];
    int64_t lo, hi;
    ora_drafter_window(p0, seq_lens[r], c->window, c->max_blocks, &lo, &hi);
    const int64_t b_lo = lo / DA_BLOCK, b_hi = hi < lo ? b_lo - 1 : hi / DA_BLOCK;
    const int64_t nparts = (b_hi - b_lo + c->part_blocks) / c->part_blocks;
    if (b_hi >= b_lo && b_hi >= c->bt_width) { rc = ORA_ERR_ARG; break; }
    for (int64_t b = b_lo; b <= b_hi; ++b) {
      const int64_t phys = block_table[(int64_t)r * c->bt_width + b];
      if (phys < 0 || phys >= num_blocks) rc = ORA_ERR_SLOT;
    }
    if (rc) break;
    for (int j = 0; j < c->q_len; ++j) {
      const int64_t m_row = (int64_t)r * c->q_len + j;
      const int64_t qp = p0 + j;
      for (int h = 0; h < DA_HEADS; ++h) {
        const uint8_t *qv = q8 + (m_row * DA_HEADS + h) * D;
        double mst = -INFINITY;
        for (int64_t i = 0; i < nparts; ++i) {
          double m = -INFINITY, l = 0.0, *o = po + i * D;
          for (int d = 0; d < D; ++d) o[d] = 0.0;
          const int64_t b_end = b_lo + (i + 1) * c->part_blocks;
          for (int64_t b = b_lo + i * c->part_blocks; b < b_end && b <= b_hi; ++b) {
            const uint8_t *blk = cache + (int64_t)block_table[(int64_t)r * c->bt_width + b] *
                                             DA_BLOCK * DA_KEY_BYTES;
            double s[DA_BLOCK], mb = -INFINITY;
            for (int k = 0; k < DA_BLOCK; ++k) {
              const int64_t kp = b * DA_BLOCK + k;
              s[k] = -INFINITY;
              if (kp < lo || kp > hi || kp <= qp - c->window) continue;
              double acc = 0.0;
              for (int d = 0; d < D; ++d) acc += lut[qv[d]] * lut[blk[k * DA_KEY_BYTES + d]];
              s[k] = acc;
              if (acc > mb) mb = acc;
            }
            const double mn = m > mb ? m : mb;
            const double ms = mn == -INFINITY ? 0.0 : mn;
            const double alpha = exp2((m - ms) * C);
            const double off = ms * C - 8.0;
            double psum = 0.0;
            for (int d = 0; d < D; ++d) o[d] *= alpha;
            for (int k = 0; k < DA_BLOCK; ++k) {
              if (s[k] == -INFINITY) continue;
              const float p = (float)exp2(s[k] * C - off);
              const double pq = lut[ora_e4m3_encode(p)];
              const uint8_t *v = blk + k * DA_KEY_BYTES + D;
              psum += (double)p;
              for (int d = 0; d < D; ++d) o[d] += pq * lut[v[d]];
            }
            l = l * alpha + psum;
            m = mn;
          }
          pm[i] = m;
          pl[i] = l;
          if (m > mst) mst = m;
        }
        double L = 0.0, acc[HEAD_DIM];
        for (int d = 0; d < D; ++d) acc[d] = 0.0;
        for (int64_t i = 0; i < nparts; ++i) {
          if (pm[i] == -INFINITY) continue;
          const double w = exp2((pm[i] - mst) * C);
          L += w * pl[i];
          for (int d = 0; d < D; ++d) acc[d] += w * po[i * D + d];
        }
        for (int d = 0; d < D; ++d) row[h * D + d] = L > 0.0 ? ora_bf16_round((float)(acc[d] / L)) : 0.0f;
      }
      for (int k = 0; k < W; ++k)
        if (out_bf16) out_bf16[m_row * W + k] = ora_bf16_encode(row[k]);
      for (int bk = 0; bk < W / 32; ++bk) {
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(row[32 * bk + i]));
        const int e = ora_mx_exponent(amax);
        for (int i = 0; i < 32; ++i)
          out_codes[m_row * W + 32 * bk + i] = ora_e4m3_encode((float)ldexp((double)row[32 * bk + i], -e));
        out_scales[m_row * (W / 32) + bk] = (uint8_t)(e + 127);
      }
    }
  }
  free(pm); free(pl); free(po); free(row);
  return rc;
}
