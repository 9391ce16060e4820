/*
 * pre_attn — GB300 (sm_103a) MiniMax-M3 sparse-layer pre-attention step.
 *
 * One call of pre_attn_run() performs, for each of M token rows:
 *   1. residual add: acc = ar + res in f32, residual_out = bf16(acc)
 *      (page "vllm.models.minimax_m3.amd.mono.kernels.pre_attn", module
 *      summary and emit_pre_attn / norm_quant);
 *   2. Gemma RMSNorm: n = acc * rsqrt(mean(acc^2) + eps) * (1 + g_in);
 *   3. activation quantisation: per-token FP8 E4M3 (scale = amax / 448, a
 *      true divide) for PA_WEIGHT_FP8_PER_CHANNEL, or MXFP8 (32-element
 *      blocks along H with E8M0 scales) for PA_WEIGHT_MXFP8;
 *   4. the fused projection y = xq . W^T (f32 accumulation) into
 *      [q x n_q | k x n_kv | v x n_kv | index_q x n_iq | index_k x 1]
 *      128-dim heads (page "vllm.models.minimax_m3.nvidia.ops.
 *      qkv_index_fused_epilogue", QkvIndexFusedEpilogueKernel: N layout);
 *   5. per head: Gemma RMSNorm + partial NeoX RoPE (rotary dim 64 of 128)
 *      on the f32 accumulator for q, k, index_q and index_k; v stays raw
 *      (pre_attn page, head_norm_rope; epilogue page, _rms_norm / _rope64);
 *   6. q and index_q outputs (bf16 and / or E4M3);
 *   7. K, V and index_k quantised and inserted into paged caches through
 *      slot_mapping: FP8 with per-token scales (pre_attn page, head tasks)
 *      or NVFP4 (epilogue page, _nvfp4_quant32 / _nvfp4_cache_views).
 * The projection y is never written to memory as a whole.
 *
 * Conventions (all entry points):
 *   - Every pointer argument that names tensor data is a DEVICE pointer owned
 *     by the caller, unless documented as host.  The library owns only its
 *     handle (host memory) and its compiled kernels.
 *   - pre_attn_run() is asynchronous on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream), allocates nothing and never
 *     synchronises.  Host-checkable argument errors return a PA_ERR_* code
 *     before anything is launched; nothing aborts.
 *   - Values that live in device memory (positions, slots) cannot be checked
 *     on the host.  The kernels skip any cache store whose slot is out of the
 *     cache's range and clamp an out-of-range position into the cos/sin
 *     table; each such event sets a bit in the workspace's status word
 *     (PA_DEV_*), read with pre_attn_device_status().
 *   - All matrices are row-major and densely packed unless a stride is given.
 *   - bf16 is IEEE binary16-brain; e4m3 is OCP FP8 E4M3 ("fn"); E8M0 is an
 *     unsigned power-of-two exponent with bias 127; E2M1 is OCP FP4.
 */
#ifndef PRE_ATTN_H
#define PRE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status */
enum pa_status {
  PA_OK = 0,
  PA_ERR_NULL = 1,        /* a required pointer is NULL */
  PA_ERR_CONFIG = 2,      /* configuration outside the supported set */
  PA_ERR_SHAPE = 3,       /* M < 0, M > max_tokens, or a size is inconsistent */
  PA_ERR_ALIGN = 4,       /* a pointer or stride violates its alignment rule */
  PA_ERR_NO_Q_OUTPUT = 5, /* neither q output requested (epilogue page asserts one) */
  PA_ERR_NO_IQ_OUTPUT = 6,/* neither index_q output requested */
  PA_ERR_ALIAS = 7,       /* residual_out overlaps ar or res (not supported) */
  PA_ERR_WORKSPACE = 8,   /* workspace NULL or smaller than pre_attn_workspace_bytes */
  PA_ERR_CUDA = 9,        /* a CUDA runtime call failed (launch, attribute, query) */
  PA_ERR_UNSUPPORTED = 10 /* a valid request this build does not implement */
};

/* Bits of the device status word (sticky until pre_attn_device_status). */
enum pa_device_status {
  PA_DEV_SLOT_RANGE = 1u << 0,  /* a slot pointed outside its cache: store skipped */
  PA_DEV_POS_RANGE = 1u << 1,   /* a position outside [0, max_pos): clamped */
  PA_DEV_WAIT_TIMEOUT = 1u << 2 /* a bounded device wait gave up (results invalid) */
};

/* ---------------------------------------------------------- formats */
enum pa_weight_format {
  /* [N, H] e4m3 + [N] f32 per-output-channel scales; activations per-token
   * FP8 (pre_attn page, GEMV tasks: "ptpc-FP8"). */
  PA_WEIGHT_FP8_PER_CHANNEL = 0,
  /* [N, H] e4m3 + E8M0 scales per 32-element K block in the F8_128x4 layout
   * (epilogue page, prepare_SF); activations MXFP8 with the same blocks. */
  PA_WEIGHT_MXFP8 = 1
};

enum pa_cache_format {
  /* Page-16 FP8 caches with per-token f32 K / V scales (pre_attn page, head
   * tasks).  Per page16 p and KV head h (page-major, head-minor):
   *   K byte (p*n_kv + h)*2048 + (d/16)*256 + t*16 + d%16   ("SHUFFLE")
   *   V byte (p*n_kv + h)*2048 + d*16 + t                     (transposed)
   *   k_scale / v_scale f32 at (p*n_kv + h)*16 + t
   * with p = page16_of(slot), t = slot % 16, d the head dim.  The index
   * cache is [num_index_slots, 128] e4m3 (unit scale) at islot*128 + d. */
  PA_CACHE_FP8 = 0,
  /* NVFP4 caches (epilogue page, _nvfp4_cache_views): the KV cache is
   * kv_pages pages of kv_page_bytes; page = slot / bs holds 2*n_kv slots of
   * bs*72 bytes (K of KV head h in slot 2h, V in slot 2h+1); within a slot,
   * token t's 128 E2M1 values take bytes t*64 + (d/64)*32 + (d%64)/2 (even
   * d in the low nibble), then the 8 E4M3 group scales (16 dims each) sit
   * after bs*64 data bytes: K and index_k linear at t*8 + g, V swizzled at
   * (t/4*4 + g/2)*8 + (g%2)*4 + t%4.  The index cache has one slot per page. */
  PA_CACHE_NVFP4 = 1
};

enum pa_flags {
  PA_FLAG_STATIC_KV_SCALE = 1 << 0, /* FP8 caches: K / V scales fixed at 1 */
  PA_FLAG_FORCE_GEMV = 1 << 1,      /* testing: the skinny path for any M <= 16 */
  PA_FLAG_FORCE_GEMM = 1 << 2,      /* testing: the tensor-core GEMM path for any M */
  PA_FLAG_NO_PDL = 1 << 3,          /* launch without programmatic dependent launch */
  PA_FLAG_GEMM_SINGLE = 1 << 4,     /* testing: tensor-core path on single CTAs (128 x 128 tiles) */
  PA_FLAG_GEMM_PAIR = 1 << 5,       /* testing: tensor-core path on CTA pairs (256 x 256 tiles) */
  PA_FLAG_FUSE = 1 << 6,            /* skinny path in one kernel (the row normalisation inside the
                                       GEMV's clusters) where the shape allows; measured slower than
                                       prologue + GEMV at the decode shape, so not the default */
  PA_FLAG_EXACT_NORM = 1 << 7,      /* testing: the many-row prologue computes every activation code
                                       from the exact normalised value (the fast path's fallback);
                                       results are bitwise the same as without it */
  PA_FLAG_GEMV_PERSIST = 1 << 9,    /* testing: the persistent skinny GEMV wherever it can run (H <= 6144),
                                       also for head counts the one-cluster-a-head grid is chosen for */
  PA_FLAG_GEMV_REGULAR = 1 << 10,   /* testing: the one-cluster-a-head skinny GEMV for any head count
                                       (not with PA_FLAG_GEMV_PERSIST) */
  PA_FLAG_TEST_WAIT_TIMEOUT = 1 << 8 /* testing: every bounded device wait gives up after 200 us
                                       instead of about a second, and the main kernel's epilogue
                                       also waits on a barrier nothing arrives on, so the wait runs
                                       out: the step's outputs and done words are not written and
                                       PA_DEV_WAIT_TIMEOUT is raised, as a real timeout would */
};

/* ----------------------------------------------------------- config */
typedef struct pa_config {
  int hidden;        /* H, the projection's K: a multiple of 128, <= 16384 */
  int n_kv_heads;    /* n_kv in {1, 2, 4} (epilogue page, kernel __init__) */
  int n_q_heads;     /* 0 -> 16 * n_kv (the pages' layout) */
  int n_iq_heads;    /* 0 -> n_kv */
  int weight_format; /* enum pa_weight_format */
  int cache_format;  /* enum pa_cache_format */
  int block_size;    /* tokens per cache page: 16 for PA_CACHE_FP8; for
                        PA_CACHE_NVFP4 a multiple of 4 (V scale swizzle) */
  int kv_page_stride;/* FP8 page16_of (pre_attn page): page-16 blocks per
                        128-token block; 0 or 8 -> page16 = slot / 16 */
  float eps;         /* RMSNorm epsilon, input and head norms */
  int max_tokens;    /* largest M pre_attn_run accepts (sizes the workspace) */
  int flags;         /* enum pa_flags */
  int gemm_grid;     /* testing: persistent GEMM grid override (0 = auto) */
} pa_config;

typedef struct pa_handle pa_handle;

/* Per-layer parameters; static across steps.  All device pointers. */
typedef struct pa_weights {
  const void *w;        /* [N, H] e4m3, row-major (K-major), N = n_heads*128 */
  const void *w_scale;  /* per-channel: [N] f32.  MXFP8: E8M0 in the
                           F8_128x4 layout of [N, H/32] (pre_attn_pack_scales) */
  const void *g_in;     /* [H] bf16 input-norm gamma */
  const void *g_q, *g_k, *g_iq, *g_ik; /* [128] bf16 head-norm gammas */
  const void *cos_sin;  /* [max_pos, 64] bf16: cos[32] | sin[32] per position */
  int64_t max_pos;
} pa_weights;

/* Per-step inputs.  All device pointers. */
typedef struct pa_step_inputs {
  const void *ar;                    /* [M, H] bf16: the all-reduce output */
  const void *res;                   /* [M, H] bf16: the residual stream */
  const int64_t *positions;          /* [M] token positions (cos_sin rows) */
  const int64_t *slot_mapping;       /* [M] KV-cache slots, -1 = skip */
  const int64_t *index_slot_mapping; /* [M] index-cache slots, -1 = skip;
                                        NULL -> slot_mapping */
} pa_step_inputs;

/* Caches, written in place at the rows' slots.  Device pointers. */
typedef struct pa_caches {
  /* PA_CACHE_FP8 */
  void *k_cache, *v_cache;      /* num_pages16 * n_kv * 2048 bytes each */
  float *k_scale, *v_scale;     /* num_pages16 * n_kv * 16 f32 each */
  void *index_cache;            /* num_index_slots * 128 bytes */
  int64_t num_pages16;
  int64_t num_index_slots;
  /* PA_CACHE_NVFP4 (base pointers and page strides: multiples of 32) */
  void *kv_cache;
  int64_t kv_pages, kv_page_bytes;   /* kv_page_bytes >= 2*n_kv*bs*72 */
  void *idx_cache;
  int64_t idx_pages, idx_page_bytes; /* idx_page_bytes >= bs*72 */
  float k_global_scale, v_global_scale; /* NVFP4 dequantisation scales (> 0) */
} pa_caches;

/* Outputs.  Device pointers; NULL = not written.  At least one q output and
 * one index_q output must be given. */
typedef struct pa_outputs {
  void *residual;   /* [M, H] bf16 = bf16(ar + res); must not overlap ar/res */
  void *q;          /* [M, n_q*128] bf16, normed + roped */
  void *q_fp8;      /* [M, n_q*128] e4m3 of q * (1 / q_fp8_scale) */
  void *iq;         /* [M, n_iq*128] bf16 index_q */
  void *iq_fp8;     /* [M, n_iq*128] e4m3 index_q, unit scale */
  float q_fp8_scale;/* dequantisation scale of q_fp8 (> 0) */
  /* Signal mode (pre_attn page, emit_pre_attn.publish_done / emit_k1's done
   * flags): NULL, or [M, n_heads] uint32 done words (4-byte aligned).  Word
   * m * n_heads + head is set to done_epoch once that (token, head) row's
   * outputs and cache bytes are written, with release semantics at GPU
   * scope: a consumer that reads done_epoch there with an acquire load (as
   * pre_attn_wait_done does) then sees every byte of the row, and the row's
   * residual.  The words are never cleared by the library: give each step a
   * new epoch (a step counter) and the consumer waits for equality.  A row
   * whose epilogue did not run (a device wait ran out) keeps its old word. */
  uint32_t *done;
  uint32_t done_epoch; /* != 0 when done is given */
} pa_outputs;

/* --------------------------------------------------------- entry points */

/* Validate `cfg` and create a handle (host memory only; no CUDA call).
 * Errors: PA_ERR_NULL, PA_ERR_CONFIG (n_kv not in {1,2,4}, H % 128 != 0 or
 * H > 16384, head counts < 1, FP8 caches with block_size != 16, NVFP4 with
 * block_size % 4 != 0, eps < 0, max_tokens < 0, unknown format). */
int pre_attn_init(const pa_config *cfg, pa_handle **out);

/* Free a handle (NULL is ignored). */
void pre_attn_destroy(pa_handle *h);

/* A static English description of a pa_status code. */
const char *pre_attn_strerror(int status);

/* The fused projection's output width N = n_heads * 128 for this handle. */
int pre_attn_out_features(const pa_handle *h);

/* Bytes of device workspace pre_attn_run needs for up to M rows (M <= the
 * handle's max_tokens): a status word and the quantised activations with
 * their scales.  Returns 0 for an invalid handle or M. */
size_t pre_attn_workspace_bytes(const pa_handle *h, int M);

/* Zero a freshly allocated workspace (cudaMemsetAsync on `stream`).  Must be
 * called once before the workspace's first pre_attn_run (the status word
 * starts clear).  Errors: PA_ERR_NULL, PA_ERR_CUDA. */
int pre_attn_workspace_init(void *workspace, size_t bytes, void *stream);

/* Bytes of the F8_128x4 layout for an [rows, hidden/32] E8M0 grid
 * (rows padded to a multiple of 128). */
size_t pre_attn_packed_scale_bytes(int rows, int hidden);

/* Re-lay a row-major [rows, hidden/32] E8M0 scale grid (device, src) into
 * the F8_128x4 layout (epilogue page, prepare_SF: [R/128, Ksf/4, 32, 4, 4])
 * that PA_WEIGHT_MXFP8 expects in pa_weights.w_scale (device, dst of
 * pre_attn_packed_scale_bytes bytes; padding rows get code 127).  Run once
 * when the weights are loaded.  Asynchronous on `stream`.
 * Errors: PA_ERR_NULL, PA_ERR_SHAPE (rows < 1, hidden % 128), PA_ERR_CUDA. */
int pre_attn_pack_scales(const void *src, void *dst, int rows, int hidden, void *stream);

/* Run the step on M rows (0 <= M <= max_tokens; M == 0 launches nothing).
 * `workspace` is a device buffer of at least pre_attn_workspace_bytes(h, M)
 * bytes, initialised once with pre_attn_workspace_init; calls that share a
 * workspace must be ordered on the GPU (one stream, or events).
 * Alignment: ar, res, residual, w, g_in and the outputs 16 bytes; NVFP4
 * cache bases and page strides 32 bytes (epilogue page, argument asserts).
 * Errors (nothing is launched): PA_ERR_NULL, PA_ERR_SHAPE, PA_ERR_ALIGN,
 * PA_ERR_NO_Q_OUTPUT, PA_ERR_NO_IQ_OUTPUT, PA_ERR_ALIAS, PA_ERR_WORKSPACE,
 * PA_ERR_CONFIG (bad cache geometry or scales); PA_ERR_CUDA if a launch
 * fails (an earlier kernel of the call may have run). */
int pre_attn_run(pa_handle *h, int M, const pa_step_inputs *in, const pa_weights *wt,
                 const pa_caches *caches, const pa_outputs *out, void *workspace,
                 size_t workspace_bytes, void *stream);

/* Read and clear the workspace's device status word (PA_DEV_* bits) into
 * *flags (host).  Synchronises `stream`.  Errors: PA_ERR_NULL, PA_ERR_CUDA. */
int pre_attn_device_status(void *workspace, uint32_t *flags, void *stream);

/* Profiling aid (the equivalent of the pre_attn page's `timeline` stamps):
 * when set, every later pre_attn_run() on this handle records `before_main`
 * and `after_main` (cudaEvent_t passed as void*; NULL = none) on its stream
 * immediately before and after the step's main kernel (the skinny GEMV or
 * the tensor-core GEMM), so cudaEventElapsedTime gives that kernel's device
 * time.  Recording between the kernels serialises them (no programmatic
 * overlap of the main kernel with the prologue), so use it for kernel timing
 * only.  The caller owns the events.  Errors: PA_ERR_NULL (h). */
int pre_attn_set_profile_events(pa_handle *h, void *before_main, void *after_main);

/* Allocation-free variant of pre_attn_run.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory and
 * so cannot supply a workspace, for example a plugin loaded into a host
 * runtime that owns all device memory through its own pool and hands none
 * out, or a process whose device memory is capped so that any cudaMalloc
 * after start-up fails.
 * It runs the same step as pre_attn_run (same arguments minus the workspace;
 * the kernels are the ones pre_attn_path(h, M) names) for 0 <= M <= 16 token
 * rows, with the kernels' scratch (status word, quantised activations and
 * their scales) in a fixed 2 MiB array inside this library; every GPU that
 * loads the library holds that array until the process exits.  It calls no
 * cudaMalloc, cudaFree or allocating library routine.
 *   - The array's device address is looked up (cudaGetSymbolAddress, with the
 *     device current) by the first call on each device, and again by the
 *     first call on a new context of that device (after cudaDeviceReset);
 *     make the first call before any stream capture.
 *   - All calls share the one array and each clears the part it uses first
 *     (cudaMemsetAsync on `stream`); calls that overlap on the GPU (other
 *     streams, other host threads) race on it, so order them.
 *   - The device status word (PA_DEV_*) of the last call on a device is read
 *     with pre_attn_noalloc_status.
 * Errors: those of pre_attn_run, and PA_ERR_SHAPE when M > 16, M > the
 * handle's max_tokens, or pre_attn_workspace_bytes(h, M) exceeds 2 MiB;
 * PA_ERR_CUDA (with pre_attn_last_cuda_error) when the lookup or the clear
 * fails. */
int pre_attn_run_noalloc(pa_handle *h, int M, const pa_step_inputs *in, const pa_weights *wt,
                         const pa_caches *caches, const pa_outputs *out, void *stream);

/* Read and clear the device status word (PA_DEV_* bits) that the last
 * pre_attn_run_noalloc on the current device left in the library's static
 * scratch, into *flags (host).  Each pre_attn_run_noalloc starts from a
 * cleared word, so the bits describe that one call.  Synchronises `stream`;
 * allocates nothing.  The pages have no counterpart (see
 * pre_attn_run_noalloc).  Errors: PA_ERR_NULL, PA_ERR_CUDA. */
int pre_attn_noalloc_status(uint32_t *flags, void *stream);

/* The consumer side of signal mode: wait on `stream` until each of the
 * `count` uint32 words at `done` (device) equals `epoch`, reading them with
 * acquire loads at GPU scope, then return (a kernel that waits and exits;
 * work queued behind it on the stream sees the rows those words cover).  It
 * may be launched with programmatic dependent launch right behind
 * pre_attn_run on the same stream: then it starts while the step's last
 * kernel runs (that kernel never waits on it) and follows the rows as they
 * are published.  Each wait is bounded by timeout_us (1 .. 10^7
 * microseconds); a word that does not reach `epoch` in time sets
 * PA_DEV_WAIT_TIMEOUT in the device word *status (device, e.g. a workspace's
 * status word, read with pre_attn_device_status) and the kernel returns.
 * Errors (nothing launched): PA_ERR_NULL, PA_ERR_SHAPE (count < 1),
 * PA_ERR_CONFIG (epoch == 0 or timeout_us out of range), PA_ERR_ALIGN;
 * PA_ERR_CUDA if the launch fails. */
int pre_attn_wait_done(const uint32_t *done, int64_t count, uint32_t epoch, uint32_t timeout_us, uint32_t *status,
                       void *stream);

/* ------------------------------------------------------ indexer scores */

/* The indexer scores that follow the step (page "vllm.models.minimax_m3.amd.
 * mono.kernels.pre_attn", emit_k1: "then every CTA's indexer scores";
 * build_pre_attn_kernel: index_scale_log2e(sm_scale) and the sparse pinned
 * init / local blocks).  The pages do not print emit_index_scores' body; this
 * is the reading: request r (r < R) owns rows m = r * q_len + i (i < q_len) at
 * positions p = seq_lens[r] - q_len + i; row m's page-128 blocks are
 * b < nb = p / 128 + 1, of which b < init_blocks and b >= nb - local_blocks
 * are pinned (attended anyway, no score); key j sits at index slot
 * block_table[r * bt_width + j / 128] * 128 + j % 128 of the FP8 index cache.
 * Row m of `scores`, columns j < nb * 128:
 *   index_scale * sum_d bf16(iq[m][head*128 + d]) * e4m3(key_j[d])  (j <= p, block not pinned)
 *   -inf                                                              (otherwise)
 * with f32 accumulation; columns from nb * 128 on are not written.  All
 * pointers are device pointers owned by the caller. */
typedef struct pa_index_args {
  const void *iq;             /* [R * q_len, iq_stride] bf16 (the step's index_q output), 8-byte aligned */
  int64_t iq_stride;          /* elements a row: a multiple of 4, >= (head + 1) * 128 */
  int head;                   /* the index_q head scored (128 dims at column head * 128) */
  const void *index_cache;    /* [num_index_slots, 128] E4M3, unit scale (PA_CACHE_FP8's index cache), 16-byte aligned */
  int64_t num_index_slots;    /* a multiple of 128 (whole page-128 blocks) */
  const int32_t *block_table; /* [R, bt_width] page-128 block ids (entries past a request's blocks unused) */
  const int32_t *seq_lens;    /* [R] tokens of each request, the step's q_len rows included */
  int R;                      /* requests, 0 .. 65535 */
  int q_len;                  /* rows a request, 1 .. 16 */
  int bt_width;               /* block-table width */
  int init_blocks;            /* pinned first blocks */
  int local_blocks;           /* pinned last blocks (the local window) */
  float index_scale;          /* pre_attn_index_scale_log2e(sm_scale) */
  float *scores;              /* [R * q_len, score_stride] f32 */
  int64_t score_stride;       /* floats a row: >= bt_width * 128 */
  uint32_t *status;           /* device status word: PA_DEV_SLOT_RANGE (a block id outside the cache, or a
                                 request shorter than q_len or longer than its block table: skipped),
                                 PA_DEV_WAIT_TIMEOUT */
  uint32_t flags;             /* 0, or PA_FLAG_TEST_WAIT_TIMEOUT (testing: every wait gives up after 200 us
                                 and the score warps also wait on a barrier nothing arrives on, so the
                                 wait runs out: the CTAs stop, their scores are not written and
                                 PA_DEV_WAIT_TIMEOUT is raised, as a real timeout would) */
} pa_index_args;

/* index_scale_log2e(sm_scale) (build_pre_attn_kernel; body not printed):
 * the reading sm_scale * log2(e), so exp2(score) = exp(sm_scale * q.k). */
float pre_attn_index_scale_log2e(float sm_scale);

/* Compute the indexer scores on `stream`.  May be launched right behind
 * pre_attn_run on the same stream: it reads the rows and keys after that
 * step's kernels complete (programmatic dependent launch).  Allocates
 * nothing, never synchronises.  Errors (nothing launched): PA_ERR_NULL,
 * PA_ERR_SHAPE, PA_ERR_CONFIG (negative block counts, NaN scale, unknown
 * flags), PA_ERR_ALIGN; PA_ERR_CUDA if the launch fails. */
int pre_attn_index_scores(const pa_index_args *args, void *stream);

/* ------------------------------------------------ the drafter's attention
 *
 * The DSpark drafter's attention (page "vllm.models.minimax_m3.amd.mono.
 * drafter.attention": module summary, qkv_rows, window, block_math /
 * block_acc, store_partial, merge_task), as three kernels on `stream`:
 *   1. q / k head norms and RoPE (qkv_rows): for each of M = R * q_len rows
 *      of the drafter's projection (16 q heads, then k, then v, 128 bf16
 *      each), q and k get the step's Gemma head RMSNorm (gammas qn, kn) and
 *      partial NeoX RoPE at positions[m]; q becomes E4M3 into q8 row
 *      m * 16 + h, k and v become E4M3 at the row's slot of the drafter
 *      cache (slot_mapping[m] < 0: not stored).  All unit scale.
 *   2. split-KV attention (3. and its merge): request r's rows sit at p0 + j
 *      (p0 = positions[r * q_len], j < q_len) and see keys kp with
 *      lo <= kp <= hi and kp > p0 + j - window, where lo = max(p0 - window
 *      + 1, 0) and hi = min(seq_lens[r] - 1, (lo / 128 + max_blocks) * 128
 *      - 1) (window); rows see each other's keys (non-causal).  The blocks
 *      lo / 128 .. hi / 128 are cut into partitions of part_blocks blocks;
 *      each partition runs an online softmax over its blocks with scores
 *      s = q . k, P = exp2(s C - (m C - 8)) (C = sm_scale * log2(e), m the
 *      running maximum), l summing P and o summing E4M3(P) V (block_acc);
 *      the partitions are merged in order, out = sum w_i o_i / sum w_i l_i
 *      with w_i = exp2((m_i - max m) C), rounded to bf16 and quantised to
 *      MXFP8 (32-value blocks along the row's 16 * 128 values, the smallest
 *      power-of-two E8M0 scale under which no value exceeds 448).  A row
 *      with no valid key gets zeros.
 * The drafter cache is page-128 blocks of 128 keys x 256 bytes (the key's
 * 128 E4M3 K bytes, then its 128 E4M3 V bytes); slot s is byte s * 256 of
 * it, block b of request r is block_table[r * bt_width + b].
 * With qkv == NULL the first kernel is skipped: q8 and the cache are taken
 * as they are.  All pointers are device pointers owned by the caller. */
typedef struct pa_drafter_args {
  const void *qkv;             /* [M, qkv_stride] bf16, or NULL; 16-byte aligned */
  int64_t qkv_stride;          /* elements a row: a multiple of 8, >= 18 * 128 */
  const void *qn, *kn;         /* [128] bf16 head-norm gammas of q and k, 16-byte aligned */
  float eps;                   /* head RMSNorm epsilon */
  const void *cos_sin;         /* [max_pos, 64] bf16 (cos of the 32 rotary pairs, then sin), 16-byte aligned */
  int64_t max_pos;             /* positions outside [0, max_pos) are clamped and flagged */
  const int64_t *positions;    /* [M]: request r's rows at positions[r * q_len] + j */
  const int64_t *slot_mapping; /* [M] drafter-cache slots of the new keys (< 0: none) */
  void *cache;                 /* [num_blocks, 128, 256] bytes, 16-byte aligned */
  int64_t num_blocks;          /* 1 .. 2^24 - 1 */
  const int32_t *block_table;  /* [R, bt_width] page-128 block ids */
  int bt_width;
  const int32_t *seq_lens;     /* [R] keys of each request, its q_len new ones included */
  int R;                       /* requests, 0 .. 65535 */
  int q_len;                   /* rows a request, 1 .. 8 (7 on the page) */
  int window;                  /* sliding window in keys (4096 on the page), >= 1 */
  int max_blocks;              /* blocks of a window at most (34 covers 4096 keys and 7 rows), >= 1 */
  int part_blocks;             /* blocks a partition: >= 1, or 0 for pre_attn_drafter_part_blocks' choice */
  float sm_scale;              /* > 0, finite: 1 / sqrt(128) on the page */
  void *q8;                    /* [M * 16, 128] E4M3: written by kernel 1 (or given), read by kernel 2;
                                  16-byte aligned */
  void *out_bf16;              /* [M, 2048] bf16 or NULL, 16-byte aligned */
  void *out_codes;             /* [M, 2048] E4M3 MXFP8 codes, 16-byte aligned */
  void *out_scales;            /* [M, 64] E8M0 scale bytes (row-major: scale k covers columns 32k .. 32k + 31) */
  void *workspace;             /* pre_attn_drafter_workspace_bytes() of scratch (the partitions' partial
                                  results), 256-byte aligned; no initial contents needed */
  size_t workspace_bytes;
  uint32_t *status;            /* device status word: PA_DEV_POS_RANGE, PA_DEV_SLOT_RANGE (a slot or block id
                                  outside the cache, or a window block past the block table: that key's store
                                  or that block skipped), PA_DEV_WAIT_TIMEOUT */
  uint32_t flags;              /* PA_FLAG_NO_PDL, PA_FLAG_TEST_WAIT_TIMEOUT */
  void *prof_before;           /* optional cudaEvent_t recorded on the stream just before the attention
                                  kernel (kernel 2), or NULL; profiling only: the record keeps kernel 2
                                  from overlapping kernel 1 */
  void *prof_after;            /* optional cudaEvent_t recorded just after kernel 2, or NULL */
} pa_drafter_args;

/* The partition length pre_attn_drafter_attention picks for part_blocks = 0:
 * max(1, floor(2 * num_sms / R)) partitions of a full window (the kernel runs
 * two CTAs an SM, so every partition of every request fits one wave),
 * max_blocks cut evenly between them: ceil(max_blocks / that).  Pure host
 * arithmetic; returns -PA_ERR_SHAPE for non-positive arguments. */
int pre_attn_drafter_part_blocks(int R, int max_blocks, int num_sms);

/* Workspace bytes of a call with these sizes (part_blocks >= 1): one
 * partial (m, l, o) of 128 rows, f32, per partition of every request.
 * Returns 0 for non-positive arguments. */
size_t pre_attn_drafter_workspace_bytes(int R, int max_blocks, int part_blocks);

/* Run the drafter's attention on `stream` (see above).  Allocates nothing,
 * never synchronises; each kernel waits for the one before it (kernel 1
 * for the previous kernel on the stream) through programmatic dependent
 * launch.
 * Errors (nothing launched): PA_ERR_NULL, PA_ERR_SHAPE, PA_ERR_CONFIG
 * (window, max_blocks or part_blocks out of range, sm_scale not positive and finite), PA_ERR_ALIGN,
 * PA_ERR_WORKSPACE; PA_ERR_CUDA if a launch fails. */
int pre_attn_drafter_attention(const pa_drafter_args *args, void *stream);

/* Main kernels a call can run (pre_attn_path). */
enum {
  PA_PATH_GEMV = 0,         /* skinny path: prologue, then the FP8 GEMV on one cluster per head */
  PA_PATH_GEMM_SINGLE = 1,  /* tensor-core path, 128 x 128 tiles on single SMs */
  PA_PATH_GEMM_PAIR = 2,    /* tensor-core path, 256 x 256 tiles on SM pairs */
  PA_PATH_GEMV_FUSED = 3,   /* skinny path in one kernel (PA_FLAG_FUSE) */
  PA_PATH_GEMV_PERSIST = 4  /* skinny path with more than four heads a resident 16-CTA cluster (H <= 6144):
                               prologue, then a persistent GEMV whose resident clusters walk the heads
                               through a 4-stage weight ring */
};

/* Which main kernel pre_attn_run(h, M, ...) launches on the current device
 * (PA_PATH_*; the choice depends on M, the handle's flags and the device's
 * SM count).  Returns a negative PA_ERR_* value for a NULL handle
 * (-PA_ERR_NULL), an M outside [1, max_tokens] or one the flags exclude
 * (-PA_ERR_SHAPE), or a failed device query (-PA_ERR_CUDA). */
int pre_attn_path(pa_handle *h, int M);

/* The last CUDA error string seen by this thread's calls ("" if none). */
const char *pre_attn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PRE_ATTN_H */
