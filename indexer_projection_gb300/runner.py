"""A torch-tensor front end of the pre-attention C-ABI.

PyTorch provides device memory and streams only; every step of the
computation runs in libpre_attn.so.  ``PreAttn`` owns a handle and a
workspace and turns tensors into the C structs of include/pre_attn.h.
"""

from __future__ import annotations

import torch

from . import binding as B


class PreAttn:
    """One configured pre-attention step (one layer's shapes and formats)."""

    def __init__(self, hidden: int, n_kv_heads: int, *, weight_format: int, cache_format: int,
                 max_tokens: int, block_size: int = 16, eps: float = 1e-6, n_q_heads: int = 0,
                 n_iq_heads: int = 0, kv_page_stride: int = 8, flags: int = 0, gemm_grid: int = 0,
                 device: torch.device | str | None = None):
        B.load()
        self.cfg = B.pa_config(hidden, n_kv_heads, n_q_heads, n_iq_heads, weight_format, cache_format,
                               block_size, kv_page_stride, eps, max_tokens, flags, gemm_grid)
        self.handle = B.pre_attn_init(self.cfg)
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.N = B.pre_attn_out_features(self.handle)
        self.ws_bytes = B.pre_attn_workspace_bytes(self.handle, max_tokens)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=self.device)
        B.pre_attn_workspace_init(self.workspace, self.ws_bytes, torch.cuda.current_stream(self.device))

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None:
            B.pre_attn_destroy(h)
            self.handle = None

    @staticmethod
    def weights(w, w_scale, g_in, g_q, g_k, g_iq, g_ik, cos_sin) -> B.pa_weights:
        return B.pa_weights(B.ptr(w), B.ptr(w_scale), B.ptr(g_in), B.ptr(g_q), B.ptr(g_k), B.ptr(g_iq),
                            B.ptr(g_ik), B.ptr(cos_sin), int(cos_sin.shape[0]))

    @staticmethod
    def fp8_caches(k_cache, v_cache, k_scale, v_scale, index_cache, num_pages16: int,
                   num_index_slots: int) -> B.pa_caches:
        c = B.pa_caches()
        c.k_cache, c.v_cache = B.ptr(k_cache), B.ptr(v_cache)
        c.k_scale, c.v_scale = B.ptr(k_scale), B.ptr(v_scale)
        c.index_cache = B.ptr(index_cache)
        c.num_pages16, c.num_index_slots = num_pages16, num_index_slots
        c.k_global_scale = c.v_global_scale = 1.0
        return c

    @staticmethod
    def nvfp4_caches(kv_cache, kv_pages: int, kv_page_bytes: int, idx_cache, idx_pages: int,
                     idx_page_bytes: int, k_global_scale: float = 1.0, v_global_scale: float = 1.0) -> B.pa_caches:
        c = B.pa_caches()
        c.kv_cache, c.kv_pages, c.kv_page_bytes = B.ptr(kv_cache), kv_pages, kv_page_bytes
        c.idx_cache, c.idx_pages, c.idx_page_bytes = B.ptr(idx_cache), idx_pages, idx_page_bytes
        c.k_global_scale, c.v_global_scale = k_global_scale, v_global_scale
        return c

    @staticmethod
    def outputs(residual=None, q=None, q_fp8=None, iq=None, iq_fp8=None, q_fp8_scale: float = 1.0, done=None,
                done_epoch: int = 0) -> B.pa_outputs:
        return B.pa_outputs(B.ptr(residual), B.ptr(q), B.ptr(q_fp8), B.ptr(iq), B.ptr(iq_fp8), q_fp8_scale,
                            B.ptr(done), done_epoch)

    def run(self, M: int, ar, res, positions, slot_mapping, weights: B.pa_weights, caches: B.pa_caches,
            outputs: B.pa_outputs, index_slot_mapping=None, stream=None, check: bool = True) -> int:
        inputs = B.pa_step_inputs(B.ptr(ar), B.ptr(res), B.ptr(positions), B.ptr(slot_mapping),
                                  B.ptr(index_slot_mapping))
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        return B.pre_attn_run(self.handle, M, inputs, weights, caches, outputs, self.workspace,
                              self.ws_bytes, stream, check=check)

    def device_status(self, stream=None) -> int:
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        return B.pre_attn_device_status(self.workspace, stream)
