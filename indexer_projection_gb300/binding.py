"""ctypes binding of the pre-attention C-ABI (include/pre_attn.h).

Argument marshalling only: the structs mirror the C structs field by field
and each function forwards to the entry point of the same name.  Pointer
fields accept None, an int device address, or any object with
``data_ptr()`` (a torch tensor); streams accept None, an int handle or an
object with ``cuda_stream``.  Loading fails loudly when libpre_attn.so is
missing: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpre_attn.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "pre_attn.h")

# enum values (include/pre_attn.h)
PA_OK, PA_ERR_NULL, PA_ERR_CONFIG, PA_ERR_SHAPE, PA_ERR_ALIGN = 0, 1, 2, 3, 4
PA_ERR_NO_Q_OUTPUT, PA_ERR_NO_IQ_OUTPUT, PA_ERR_ALIAS, PA_ERR_WORKSPACE = 5, 6, 7, 8
PA_ERR_CUDA, PA_ERR_UNSUPPORTED = 9, 10
PA_DEV_SLOT_RANGE, PA_DEV_POS_RANGE, PA_DEV_WAIT_TIMEOUT = 1, 2, 4
PA_WEIGHT_FP8_PER_CHANNEL, PA_WEIGHT_MXFP8 = 0, 1
PA_CACHE_FP8, PA_CACHE_NVFP4 = 0, 1
PA_FLAG_STATIC_KV_SCALE, PA_FLAG_FORCE_GEMV, PA_FLAG_FORCE_GEMM, PA_FLAG_NO_PDL = 1, 2, 4, 8
PA_FLAG_GEMM_SINGLE, PA_FLAG_GEMM_PAIR, PA_FLAG_FUSE, PA_FLAG_EXACT_NORM = 16, 32, 64, 128
PA_FLAG_TEST_WAIT_TIMEOUT = 256
PA_FLAG_GEMV_PERSIST, PA_FLAG_GEMV_REGULAR = 512, 1024
PA_PATH_GEMV, PA_PATH_GEMM_SINGLE, PA_PATH_GEMM_PAIR, PA_PATH_GEMV_FUSED, PA_PATH_GEMV_PERSIST = 0, 1, 2, 3, 4

_vp = ctypes.c_void_p


class pa_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("n_q_heads", ctypes.c_int),
                ("n_iq_heads", ctypes.c_int), ("weight_format", ctypes.c_int),
                ("cache_format", ctypes.c_int), ("block_size", ctypes.c_int),
                ("kv_page_stride", ctypes.c_int), ("eps", ctypes.c_float),
                ("max_tokens", ctypes.c_int), ("flags", ctypes.c_int), ("gemm_grid", ctypes.c_int)]


class pa_weights(ctypes.Structure):
    _fields_ = [("w", _vp), ("w_scale", _vp), ("g_in", _vp), ("g_q", _vp), ("g_k", _vp),
                ("g_iq", _vp), ("g_ik", _vp), ("cos_sin", _vp), ("max_pos", ctypes.c_int64)]


class pa_step_inputs(ctypes.Structure):
    _fields_ = [("ar", _vp), ("res", _vp), ("positions", _vp), ("slot_mapping", _vp),
                ("index_slot_mapping", _vp)]


class pa_caches(ctypes.Structure):
    _fields_ = [("k_cache", _vp), ("v_cache", _vp), ("k_scale", _vp), ("v_scale", _vp),
                ("index_cache", _vp), ("num_pages16", ctypes.c_int64),
                ("num_index_slots", ctypes.c_int64), ("kv_cache", _vp), ("kv_pages", ctypes.c_int64),
                ("kv_page_bytes", ctypes.c_int64), ("idx_cache", _vp), ("idx_pages", ctypes.c_int64),
                ("idx_page_bytes", ctypes.c_int64), ("k_global_scale", ctypes.c_float),
                ("v_global_scale", ctypes.c_float)]


class pa_outputs(ctypes.Structure):
    _fields_ = [("residual", _vp), ("q", _vp), ("q_fp8", _vp), ("iq", _vp), ("iq_fp8", _vp),
                ("q_fp8_scale", ctypes.c_float), ("done", _vp), ("done_epoch", ctypes.c_uint32)]


class pa_index_args(ctypes.Structure):
    _fields_ = [("iq", _vp), ("iq_stride", ctypes.c_int64), ("head", ctypes.c_int), ("index_cache", _vp),
                ("num_index_slots", ctypes.c_int64), ("block_table", _vp), ("seq_lens", _vp), ("R", ctypes.c_int),
                ("q_len", ctypes.c_int), ("bt_width", ctypes.c_int), ("init_blocks", ctypes.c_int),
                ("local_blocks", ctypes.c_int), ("index_scale", ctypes.c_float), ("scores", _vp),
                ("score_stride", ctypes.c_int64), ("status", _vp), ("flags", ctypes.c_uint32)]


class pa_drafter_args(ctypes.Structure):
    _fields_ = [("qkv", _vp), ("qkv_stride", ctypes.c_int64), ("qn", _vp), ("kn", _vp), ("eps", ctypes.c_float),
                ("cos_sin", _vp), ("max_pos", ctypes.c_int64), ("positions", _vp), ("slot_mapping", _vp),
                ("cache", _vp), ("num_blocks", ctypes.c_int64), ("block_table", _vp), ("bt_width", ctypes.c_int),
                ("seq_lens", _vp), ("R", ctypes.c_int), ("q_len", ctypes.c_int), ("window", ctypes.c_int),
                ("max_blocks", ctypes.c_int), ("part_blocks", ctypes.c_int), ("sm_scale", ctypes.c_float),
                ("q8", _vp), ("out_bf16", _vp), ("out_codes", _vp), ("out_scales", _vp), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t), ("status", _vp), ("flags", ctypes.c_uint32),
                ("prof_before", _vp), ("prof_after", _vp)]


class PreAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({pre_attn_strerror(status)})")


_lib = None


def load(path: str = LIB_PATH):
    """Load libpre_attn.so (raises if it is missing or lacks a symbol)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} not built: the pre-attention CUDA library is required")
    L = ctypes.CDLL(path)
    sz, i, u32p = ctypes.c_size_t, ctypes.c_int, ctypes.POINTER(ctypes.c_uint32)
    H = ctypes.c_void_p
    sigs = {
        "pre_attn_init": (i, [ctypes.POINTER(pa_config), ctypes.POINTER(H)]),
        "pre_attn_destroy": (None, [H]),
        "pre_attn_strerror": (ctypes.c_char_p, [i]),
        "pre_attn_out_features": (i, [H]),
        "pre_attn_workspace_bytes": (sz, [H, i]),
        "pre_attn_workspace_init": (i, [_vp, sz, _vp]),
        "pre_attn_packed_scale_bytes": (sz, [i, i]),
        "pre_attn_pack_scales": (i, [_vp, _vp, i, i, _vp]),
        "pre_attn_run": (i, [H, i, ctypes.POINTER(pa_step_inputs), ctypes.POINTER(pa_weights),
                             ctypes.POINTER(pa_caches), ctypes.POINTER(pa_outputs), _vp, sz, _vp]),
        "pre_attn_device_status": (i, [_vp, u32p, _vp]),
        "pre_attn_last_cuda_error": (ctypes.c_char_p, []),
        "pre_attn_path": (i, [H, i]),
        "pre_attn_set_profile_events": (i, [H, _vp, _vp]),
        "pre_attn_run_noalloc": (i, [H, i, ctypes.POINTER(pa_step_inputs), ctypes.POINTER(pa_weights),
                                     ctypes.POINTER(pa_caches), ctypes.POINTER(pa_outputs), _vp]),
        "pre_attn_noalloc_status": (i, [u32p, _vp]),
        "pre_attn_wait_done": (i, [_vp, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint32, _vp, _vp]),
        "pre_attn_index_scale_log2e": (ctypes.c_float, [ctypes.c_float]),
        "pre_attn_index_scores": (i, [ctypes.POINTER(pa_index_args), _vp]),
        "pre_attn_drafter_part_blocks": (i, [i, i, i]),
        "pre_attn_drafter_workspace_bytes": (sz, [i, i, i]),
        "pre_attn_drafter_attention": (i, [ctypes.POINTER(pa_drafter_args), _vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def declared_symbols(header: str = HEADER) -> list[str]:
    """The entry points include/pre_attn.h declares."""
    with open(header) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(pre_attn_\w+)\s*\(", text)))


def ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def stream_ptr(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def pre_attn_strerror(status: int) -> str:
    return load().pre_attn_strerror(int(status)).decode()


def pre_attn_last_cuda_error() -> str:
    return load().pre_attn_last_cuda_error().decode()


def pre_attn_init(cfg: pa_config) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    st = load().pre_attn_init(ctypes.byref(cfg), ctypes.byref(h))
    if st != PA_OK:
        raise PreAttnError(st, "pre_attn_init")
    return h


def pre_attn_destroy(h) -> None:
    load().pre_attn_destroy(h)


def pre_attn_out_features(h) -> int:
    return load().pre_attn_out_features(h)


def pre_attn_path(h, M: int) -> int:
    """PA_PATH_* of the main kernel a call with M rows launches."""
    st = load().pre_attn_path(h, int(M))
    if st < 0:
        raise PreAttnError(-st, "pre_attn_path")
    return st


def pre_attn_workspace_bytes(h, M: int) -> int:
    return load().pre_attn_workspace_bytes(h, int(M))


def pre_attn_workspace_init(workspace, nbytes: int, stream=None) -> None:
    st = load().pre_attn_workspace_init(ptr(workspace), int(nbytes), stream_ptr(stream))
    if st != PA_OK:
        raise PreAttnError(st, "pre_attn_workspace_init")


def pre_attn_packed_scale_bytes(rows: int, hidden: int) -> int:
    return load().pre_attn_packed_scale_bytes(int(rows), int(hidden))


def pre_attn_pack_scales(src, dst, rows: int, hidden: int, stream=None) -> None:
    st = load().pre_attn_pack_scales(ptr(src), ptr(dst), int(rows), int(hidden), stream_ptr(stream))
    if st != PA_OK:
        raise PreAttnError(st, "pre_attn_pack_scales")


def pre_attn_run(h, M: int, inputs: pa_step_inputs, weights: pa_weights, caches: pa_caches,
                 outputs: pa_outputs, workspace, workspace_bytes: int, stream=None,
                 check: bool = True) -> int:
    st = load().pre_attn_run(h, int(M), ctypes.byref(inputs), ctypes.byref(weights),
                             ctypes.byref(caches), ctypes.byref(outputs), ptr(workspace),
                             int(workspace_bytes), stream_ptr(stream))
    if check and st != PA_OK:
        extra = pre_attn_last_cuda_error() if st == PA_ERR_CUDA else ""
        raise PreAttnError(st, "pre_attn_run " + extra)
    return st


def pre_attn_run_noalloc(h, M: int, inputs: pa_step_inputs, weights: pa_weights, caches: pa_caches,
                         outputs: pa_outputs, stream=None, check: bool = True) -> int:
    st = load().pre_attn_run_noalloc(h, int(M), ctypes.byref(inputs), ctypes.byref(weights),
                                     ctypes.byref(caches), ctypes.byref(outputs), stream_ptr(stream))
    if check and st != PA_OK:
        extra = pre_attn_last_cuda_error() if st == PA_ERR_CUDA else ""
        raise PreAttnError(st, "pre_attn_run_noalloc " + extra)
    return st


def pre_attn_noalloc_status(stream=None) -> int:
    """PA_DEV_* bits of the last pre_attn_run_noalloc on the current device (read and cleared)."""
    v = ctypes.c_uint32(0)
    st = load().pre_attn_noalloc_status(ctypes.byref(v), stream_ptr(stream))
    if st != PA_OK:
        raise PreAttnError(st, "pre_attn_noalloc_status " + (pre_attn_last_cuda_error() if st == PA_ERR_CUDA else ""))
    return int(v.value)


def pre_attn_set_profile_events(h, before_main=None, after_main=None) -> None:
    """Events (torch.cuda.Event or raw cudaEvent_t ints) recorded around the main kernel."""
    def ev(e):
        if e is None or isinstance(e, int):
            return e
        return int(e.cuda_event)
    st = load().pre_attn_set_profile_events(h, ev(before_main), ev(after_main))
    if st != PA_OK:
        raise PreAttnError(st, "pre_attn_set_profile_events")


def pre_attn_wait_done(done, count: int, epoch: int, timeout_us: int, status, stream=None, check: bool = True) -> int:
    st = load().pre_attn_wait_done(ptr(done), int(count), int(epoch), int(timeout_us), ptr(status), stream_ptr(stream))
    if check and st != PA_OK:
        raise PreAttnError(st, "pre_attn_wait_done " + (pre_attn_last_cuda_error() if st == PA_ERR_CUDA else ""))
    return st


def pre_attn_index_scale_log2e(sm_scale: float) -> float:
    return load().pre_attn_index_scale_log2e(float(sm_scale))


def pre_attn_index_scores(args: pa_index_args, stream=None, check: bool = True) -> int:
    st = load().pre_attn_index_scores(ctypes.byref(args), stream_ptr(stream))
    if check and st != PA_OK:
        raise PreAttnError(st, "pre_attn_index_scores " + (pre_attn_last_cuda_error() if st == PA_ERR_CUDA else ""))
    return st


def pre_attn_drafter_part_blocks(R: int, max_blocks: int, num_sms: int) -> int:
    return int(load().pre_attn_drafter_part_blocks(int(R), int(max_blocks), int(num_sms)))


def pre_attn_drafter_workspace_bytes(R: int, max_blocks: int, part_blocks: int) -> int:
    return int(load().pre_attn_drafter_workspace_bytes(int(R), int(max_blocks), int(part_blocks)))


def pre_attn_drafter_attention(args: pa_drafter_args, stream=None, check: bool = True) -> int:
    st = load().pre_attn_drafter_attention(ctypes.byref(args), stream_ptr(stream))
    if check and st != PA_OK:
        raise PreAttnError(st, "pre_attn_drafter_attention " +
                           (pre_attn_last_cuda_error() if st == PA_ERR_CUDA else ""))
    return st


def pre_attn_device_status(workspace, stream=None) -> int:
    v = ctypes.c_uint32(0)
    st = load().pre_attn_device_status(ptr(workspace), ctypes.byref(v), stream_ptr(stream))
    if st != PA_OK:
        raise PreAttnError(st, "pre_attn_device_status")
    return int(v.value)
