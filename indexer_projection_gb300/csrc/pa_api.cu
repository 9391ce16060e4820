// The C-ABI of the pre-attention step (declared in include/pre_attn.h):
// configuration checks, workspace layout, host-side argument validation and
// the launch sequence prologue -> (skinny GEMV | tcgen05 GEMM), chained with
// programmatic dependent launch on the caller's stream.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "../../include/pre_attn.h"
#include "pa_device.cuh"
#include "pa_launch.h"

struct pa_handle {
  pa_config cfg;
  int n_q, n_kv, n_iq, n_heads, N;
  int device;   // device of the cached SM count (-1: not queried yet)
  int num_sms;
  int64_t l2_bytes;
  int early_max[2];  // many-row prologue (256 / 1024 threads a CTA): the largest grid resident
                     // at once with at most two CTAs an SM (it then triggers the GEMM early)
  cudaEvent_t prof_before, prof_after;  // optional events around the main kernel
};

namespace {

thread_local char g_cuda_err[256] = "";

int cuda_fail(cudaError_t e) {
  snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return PA_ERR_CUDA;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool uses_gemv(const pa_config &c, int M) {
  return (c.flags & PA_FLAG_FORCE_GEMV) ? true : (c.flags & PA_FLAG_FORCE_GEMM) ? false : M <= 16;
}

// Workspace layout for M rows.  The status word sits at offset 0 and carries
// state between calls (PA_DEV_* bits, sticky until read); the rest is
// scratch: the prologue's quantised activations and their scales.
struct WsLayout {
  size_t status, x_scale, xsf, xq, total;
  int m_pad;
};

WsLayout ws_layout(const pa_handle *h, int M) {
  WsLayout L;
  const size_t H = (size_t)h->cfg.hidden;
  L.m_pad = (M + 127) / 128 * 128;
  L.status = 0;
  size_t off = 256;
  L.x_scale = off;
  off = align_up(off + sizeof(float) * (size_t)(M > 0 ? M : 1), 256);
  L.xsf = off;
  if (h->cfg.weight_format == PA_WEIGHT_MXFP8)  // the MXFP8 activation scales
    off = align_up(off + (size_t)(L.m_pad > 0 ? L.m_pad : 128) * (H / 32), 256);
  L.xq = off;
  off = align_up(off + (size_t)M * H, 256);
  L.total = off;
  return L;
}

// The device's SM count, queried once per device.
cudaError_t query_sms(pa_handle *h) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (h->device != dev) {
    int sms = 0, l2 = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess) return e;
    h->num_sms = sms;
    h->l2_bytes = l2;
    for (int wide = 0; wide < 2; ++wide) {
      int per_sm = 0;
      e = pa::prologue_ctas_per_sm(h->cfg.hidden, h->cfg.weight_format == PA_WEIGHT_MXFP8 ? 1 : 0, wide != 0, &per_sm);
      if (e != cudaSuccess) return e;
      h->early_max[wide] = (per_sm < 2 ? per_sm : 2) * sms;
    }
    h->device = dev;
  }
  return cudaSuccess;
}


// Main kernel for M rows (h->num_sms known; the skinny path's fusion check
// queries the device once).  256 x 256 pair tiles cost about 1.5x a
// 128 x 128 tile on one SM: the pairs are used unless wave quantisation
// favours the finer tiles.
int choose_path(const pa_handle *h, int M) {
  const pa_config &c = h->cfg;
  if (uses_gemv(c, M)) {
    if ((c.flags & PA_FLAG_FUSE) && pa::gemv_fuses_prologue(c.hidden, c.weight_format)) return PA_PATH_GEMV_FUSED;
    // more heads than clusters of the regular grid fit at once: the persistent GEMV
    if (!(c.flags & PA_FLAG_GEMV_REGULAR) &&
        pa::gemv_persist_clusters(h->N / 128, c.hidden, c.weight_format, (c.flags & PA_FLAG_GEMV_PERSIST) != 0) > 0)
      return PA_PATH_GEMV_PERSIST;
    return PA_PATH_GEMV;
  }
  if (c.flags & PA_FLAG_GEMM_SINGLE) return PA_PATH_GEMM_SINGLE;
  if (c.flags & PA_FLAG_GEMM_PAIR) return PA_PATH_GEMM_PAIR;
  const int sms = h->num_sms > 1 ? h->num_sms : 2;
  const int64_t t1 = (int64_t)((M + 127) / 128) * (h->N / 128);
  const int64_t t2 = (int64_t)((M + 255) / 256) * ((h->N + 255) / 256);
  const int64_t w1 = (t1 + sms - 1) / sms;
  const int64_t w2 = (t2 + sms / 2 - 1) / (sms / 2);
  return 3 * w2 <= 2 * w1 ? PA_PATH_GEMM_PAIR : PA_PATH_GEMM_SINGLE;
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

namespace pa {
int record_cuda_error(cudaError_t e) { return cuda_fail(e); }
}  // namespace pa

extern "C" {

const char *pre_attn_strerror(int s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "a required pointer is NULL";
    case PA_ERR_CONFIG: return "configuration outside the supported set";
    case PA_ERR_SHAPE: return "M or a size is out of range";
    case PA_ERR_ALIGN: return "a pointer or stride violates its alignment rule";
    case PA_ERR_NO_Q_OUTPUT: return "no q output requested (need q and/or q_fp8)";
    case PA_ERR_NO_IQ_OUTPUT: return "no index_q output requested (need iq and/or iq_fp8)";
    case PA_ERR_ALIAS: return "residual partially overlaps ar or res";
    case PA_ERR_WORKSPACE: return "workspace NULL or too small";
    case PA_ERR_CUDA: return "a CUDA runtime call failed";
    case PA_ERR_UNSUPPORTED: return "valid request not implemented by this build";
    default: return "unknown status";
  }
}

const char *pre_attn_last_cuda_error(void) { return g_cuda_err; }

int pre_attn_path(pa_handle *h, int M) {
  if (!h) return -PA_ERR_NULL;
  if (M < 1 || M > h->cfg.max_tokens) return -PA_ERR_SHAPE;
  if (uses_gemv(h->cfg, M) && M > 16) return -PA_ERR_SHAPE;
  const cudaError_t e = query_sms(h);
  if (e != cudaSuccess) return -cuda_fail(e);
  return choose_path(h, M);
}

int pre_attn_init(const pa_config *cfg, pa_handle **out) {
  if (!cfg || !out) return PA_ERR_NULL;
  *out = nullptr;
  const pa_config &c = *cfg;
  if (c.hidden <= 0 || c.hidden % 128 || c.hidden > 16384) return PA_ERR_CONFIG;
  if (c.n_kv_heads != 1 && c.n_kv_heads != 2 && c.n_kv_heads != 4) return PA_ERR_CONFIG;
  if (c.n_q_heads < 0 || c.n_iq_heads < 0) return PA_ERR_CONFIG;
  if (c.weight_format != PA_WEIGHT_FP8_PER_CHANNEL && c.weight_format != PA_WEIGHT_MXFP8) return PA_ERR_CONFIG;
  if (c.cache_format == PA_CACHE_FP8) {
    if (c.block_size != 16) return PA_ERR_CONFIG;
    if (c.kv_page_stride < 0) return PA_ERR_CONFIG;
  } else if (c.cache_format == PA_CACHE_NVFP4) {
    if (c.block_size < 4 || c.block_size % 4 || c.block_size > 1024) return PA_ERR_CONFIG;
  } else {
    return PA_ERR_CONFIG;
  }
  if (!(c.eps >= 0.0f) || c.max_tokens < 0 || c.gemm_grid < 0) return PA_ERR_CONFIG;
  if ((c.flags & PA_FLAG_FORCE_GEMV) && (c.flags & PA_FLAG_FORCE_GEMM)) return PA_ERR_CONFIG;
  if ((c.flags & PA_FLAG_GEMM_SINGLE) && (c.flags & PA_FLAG_GEMM_PAIR)) return PA_ERR_CONFIG;
  if ((c.flags & PA_FLAG_GEMV_PERSIST) && (c.flags & PA_FLAG_GEMV_REGULAR)) return PA_ERR_CONFIG;
  pa_handle *h = new (std::nothrow) pa_handle;
  if (!h) return PA_ERR_CONFIG;
  h->cfg = c;
  h->n_kv = c.n_kv_heads;
  h->n_q = c.n_q_heads ? c.n_q_heads : 16 * c.n_kv_heads;
  h->n_iq = c.n_iq_heads ? c.n_iq_heads : c.n_kv_heads;
  h->n_heads = h->n_q + 2 * h->n_kv + h->n_iq + 1;
  h->N = h->n_heads * 128;
  if (h->cfg.kv_page_stride == 0) h->cfg.kv_page_stride = 8;
  h->device = -1;
  h->num_sms = 0;
  h->l2_bytes = 0;
  h->early_max[0] = h->early_max[1] = 0;
  h->prof_before = h->prof_after = nullptr;
  *out = h;
  return PA_OK;
}

void pre_attn_destroy(pa_handle *h) { delete h; }

int pre_attn_out_features(const pa_handle *h) { return h ? h->N : 0; }

int pre_attn_set_profile_events(pa_handle *h, void *before_main, void *after_main) {
  if (!h) return PA_ERR_NULL;
  h->prof_before = static_cast<cudaEvent_t>(before_main);
  h->prof_after = static_cast<cudaEvent_t>(after_main);
  return PA_OK;
}

size_t pre_attn_workspace_bytes(const pa_handle *h, int M) {
  if (!h || M < 0 || M > h->cfg.max_tokens) return 0;
  return ws_layout(h, M).total;
}

int pre_attn_workspace_init(void *workspace, size_t bytes, void *stream) {
  if (!workspace) return PA_ERR_NULL;
  cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream);
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

size_t pre_attn_packed_scale_bytes(int rows, int hidden) {
  if (rows < 1 || hidden < 128 || hidden % 128) return 0;
  return (size_t)((rows + 127) / 128 * 128) * (size_t)(hidden / 32);
}

int pre_attn_pack_scales(const void *src, void *dst, int rows, int hidden, void *stream) {
  if (!src || !dst) return PA_ERR_NULL;
  if (rows < 1 || hidden < 128 || hidden % 128) return PA_ERR_SHAPE;
  cudaError_t e = pa::launch_pack_scales(static_cast<const uint8_t *>(src), static_cast<uint8_t *>(dst), rows,
                                         hidden / 32, (cudaStream_t)stream);
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int pre_attn_device_status(void *workspace, uint32_t *flags, void *stream) {
  if (!workspace || !flags) return PA_ERR_NULL;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(v), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  *flags = v;
  return PA_OK;
}

int pre_attn_run(pa_handle *h, int M, const pa_step_inputs *in, const pa_weights *wt, const pa_caches *cc,
                 const pa_outputs *out, void *workspace, size_t workspace_bytes, void *stream) {
  if (!h || !in || !wt || !cc || !out) return PA_ERR_NULL;
  const pa_config &c = h->cfg;
  if (M < 0 || M > c.max_tokens) return PA_ERR_SHAPE;
  if (!workspace) return PA_ERR_WORKSPACE;
  const WsLayout L = ws_layout(h, M);
  if (workspace_bytes < L.total) return PA_ERR_WORKSPACE;
  if (!out->q && !out->q_fp8) return PA_ERR_NO_Q_OUTPUT;
  if (!out->iq && !out->iq_fp8) return PA_ERR_NO_IQ_OUTPUT;
  if (!in->ar || !in->res || !in->positions || !in->slot_mapping) return PA_ERR_NULL;
  if (!wt->w || !wt->w_scale || !wt->g_in || !wt->g_q || !wt->g_k || !wt->g_iq || !wt->g_ik || !wt->cos_sin)
    return PA_ERR_NULL;
  if (wt->max_pos < 1) return PA_ERR_SHAPE;
  const bool fp8c = c.cache_format == PA_CACHE_FP8;
  if (fp8c) {
    if (!cc->k_cache || !cc->v_cache || !cc->k_scale || !cc->v_scale || !cc->index_cache) return PA_ERR_NULL;
    if (cc->num_pages16 < 1 || cc->num_index_slots < 1) return PA_ERR_CONFIG;
  } else {
    if (!cc->kv_cache || !cc->idx_cache) return PA_ERR_NULL;
    const int64_t slot_bytes = (int64_t)c.block_size * 72;
    if (cc->kv_pages < 1 || cc->idx_pages < 1) return PA_ERR_CONFIG;
    if (cc->kv_page_bytes < 2 * h->n_kv * slot_bytes || cc->idx_page_bytes < slot_bytes) return PA_ERR_CONFIG;
    if (cc->kv_page_bytes % 32 || cc->idx_page_bytes % 32) return PA_ERR_ALIGN;
    if (!aligned(cc->kv_cache, 32) || !aligned(cc->idx_cache, 32)) return PA_ERR_ALIGN;
    if (!(cc->k_global_scale > 0.0f) || !(cc->v_global_scale > 0.0f)) return PA_ERR_CONFIG;
  }
  if (out->q_fp8 && !(out->q_fp8_scale > 0.0f)) return PA_ERR_CONFIG;
  if (out->done && out->done_epoch == 0) return PA_ERR_CONFIG;
  if (out->done && !aligned(out->done, 4)) return PA_ERR_ALIGN;
  // alignment (16-byte vector accesses; 256 for the workspace)
  const void *a16[] = {in->ar, in->res, out->residual, wt->w, wt->w_scale, wt->g_in, wt->g_q, wt->g_k,
                       wt->g_iq, wt->g_ik, wt->cos_sin, out->q, out->q_fp8, out->iq, out->iq_fp8,
                       fp8c ? cc->k_cache : nullptr, fp8c ? cc->v_cache : nullptr,
                       fp8c ? cc->index_cache : nullptr};
  for (const void *p : a16)
    if (p && !aligned(p, 16)) return PA_ERR_ALIGN;
  if (fp8c && (!aligned(cc->k_scale, 4) || !aligned(cc->v_scale, 4))) return PA_ERR_ALIGN;
  if (!aligned(in->positions, 8) || !aligned(in->slot_mapping, 8) ||
      (in->index_slot_mapping && !aligned(in->index_slot_mapping, 8)))
    return PA_ERR_ALIGN;
  if (!aligned(workspace, 256)) return PA_ERR_ALIGN;
  // residual: separate, or exactly in place over ar or res (each element is
  // read and then written by the same thread)
  const size_t act_bytes = (size_t)M * c.hidden * 2;
  if (out->residual) {
    for (const void *src : {in->ar, in->res})
      if (out->residual != src && ranges_overlap(out->residual, act_bytes, src, act_bytes)) return PA_ERR_ALIAS;
  }
  const bool gemv = uses_gemv(c, M);
  if (gemv && M > 16) return PA_ERR_SHAPE;
  if (M == 0) return PA_OK;

  cudaError_t e = query_sms(h);
  if (e != cudaSuccess) return cuda_fail(e);
  const int path = choose_path(h, M);

  pa::Params p;
  memset(&p, 0, sizeof(p));
  p.M = M;
  p.H = c.hidden;
  p.N = h->N;
  p.n_heads = h->n_heads;
  p.n_q = h->n_q;
  p.n_kv = h->n_kv;
  p.n_iq = h->n_iq;
  p.k0 = h->n_q;
  p.v0 = p.k0 + h->n_kv;
  p.iq0 = p.v0 + h->n_kv;
  p.ik0 = p.iq0 + h->n_iq;
  p.weight_fmt = c.weight_format;
  p.cache_fmt = c.cache_format;
  p.bs = c.block_size;
  p.kps = c.kv_page_stride;
  p.static_kv = (c.flags & PA_FLAG_STATIC_KV_SCALE) ? 1 : 0;
  p.exact_norm = (c.flags & PA_FLAG_EXACT_NORM) ? 1 : 0;
  p.eps = c.eps;
  p.ar = static_cast<const __nv_bfloat16 *>(in->ar);
  p.res = static_cast<const __nv_bfloat16 *>(in->res);
  p.g_in = static_cast<const __nv_bfloat16 *>(wt->g_in);
  p.w = static_cast<const uint8_t *>(wt->w);
  if (c.weight_format == PA_WEIGHT_FP8_PER_CHANNEL) p.w_scale = static_cast<const float *>(wt->w_scale);
  else p.wsf = static_cast<const uint8_t *>(wt->w_scale);
  p.g_q = static_cast<const __nv_bfloat16 *>(wt->g_q);
  p.g_k = static_cast<const __nv_bfloat16 *>(wt->g_k);
  p.g_iq = static_cast<const __nv_bfloat16 *>(wt->g_iq);
  p.g_ik = static_cast<const __nv_bfloat16 *>(wt->g_ik);
  p.cos_sin = static_cast<const __nv_bfloat16 *>(wt->cos_sin);
  p.max_pos = wt->max_pos;
  p.pos = in->positions;
  p.slot = in->slot_mapping;
  p.islot = in->index_slot_mapping ? in->index_slot_mapping : in->slot_mapping;
  if (fp8c) {
    p.k_cache = static_cast<uint8_t *>(cc->k_cache);
    p.v_cache = static_cast<uint8_t *>(cc->v_cache);
    p.index_cache = static_cast<uint8_t *>(cc->index_cache);
    p.k_scale = cc->k_scale;
    p.v_scale = cc->v_scale;
    p.num_pages16 = cc->num_pages16;
    p.num_index_slots = cc->num_index_slots;
  } else {
    p.kv_cache = static_cast<uint8_t *>(cc->kv_cache);
    p.idx_cache = static_cast<uint8_t *>(cc->idx_cache);
    p.kv_pages = cc->kv_pages;
    p.kv_page_bytes = cc->kv_page_bytes;
    p.idx_pages = cc->idx_pages;
    p.idx_page_bytes = cc->idx_page_bytes;
    p.k_gs_inv = 1.0f / cc->k_global_scale;
    p.v_gs_inv = 1.0f / cc->v_global_scale;
  }
  p.residual = static_cast<__nv_bfloat16 *>(out->residual);
  p.q = static_cast<__nv_bfloat16 *>(out->q);
  p.iq = static_cast<__nv_bfloat16 *>(out->iq);
  p.q_fp8 = static_cast<uint8_t *>(out->q_fp8);
  p.iq_fp8 = static_cast<uint8_t *>(out->iq_fp8);
  p.q_fp8_inv = out->q_fp8 ? 1.0f / out->q_fp8_scale : 1.0f;
  p.done = out->done;
  p.done_epoch = out->done_epoch;
  p.test_timeout = (c.flags & PA_FLAG_TEST_WAIT_TIMEOUT) ? 1 : 0;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  p.status = reinterpret_cast<uint32_t *>(ws + L.status);
  p.x_scale = reinterpret_cast<float *>(ws + L.x_scale);
  p.xsf = ws + L.xsf;
  p.xq = ws + L.xq;
  p.m_pad = L.m_pad;

  const bool pdl = !(c.flags & PA_FLAG_NO_PDL);
  cudaStream_t s = (cudaStream_t)stream;
  // the skinny path normalises the rows inside its own launch when it can
  const bool fused = path == PA_PATH_GEMV_FUSED;
  if (gemv && !fused) {
    e = pa::launch_prologue_rows(p, pdl, s);
    if (e != cudaSuccess) return cuda_fail(e);
  } else if (!gemv) {
    const int grid = c.weight_format == PA_WEIGHT_MXFP8 ? L.m_pad : M;
    e = pa::launch_prologue(p, grid, pdl, h->early_max[grid <= 64 ? 1 : 0], s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (h->prof_before && (e = cudaEventRecord(h->prof_before, s)) != cudaSuccess) return cuda_fail(e);
  if (path == PA_PATH_GEMV_PERSIST) {
    const int clusters = pa::gemv_persist_clusters(h->N / 128, c.hidden, c.weight_format,
                                                   (c.flags & PA_FLAG_GEMV_PERSIST) != 0);
    e = clusters > 0 ? pa::launch_gemv_persist(p, clusters, pdl, s) : cudaErrorNotSupported;
  } else if (gemv) {
    e = pa::launch_gemv(p, fused, pdl, s);
  } else {
    e = path == PA_PATH_GEMM_PAIR ? pa::launch_gemm_pair(p, h->num_sms, h->l2_bytes, c.gemm_grid, pdl, s)
                                  : pa::launch_gemm(p, h->num_sms, c.gemm_grid, pdl, s);
  }
  if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return cuda_fail(e);
  if (h->prof_after && (e = cudaEventRecord(h->prof_after, s)) != cudaSuccess) return cuda_fail(e);
  return PA_OK;
}

}  // extern "C"
