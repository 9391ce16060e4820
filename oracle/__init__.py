"""Test infrastructure: ctypes wrapper around the plain-C CPU oracle.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package.  The product path (the CUDA library
and its binding) never touches it, and it never touches the product path.

The oracle restates the MiniMax-M3 sparse-layer pre-attention step from the
pages "vllm.models.minimax_m3.amd.mono.kernels.pre_attn" (K1 mono_pre) and
"vllm.models.minimax_m3.nvidia.ops.qkv_index_fused_epilogue", and the DSpark
drafter's attention from "vllm.models.minimax_m3.amd.mono.drafter.attention";
each C function cites the symbol it follows.
"""

from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pre_attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

HEAD_DIM = 128


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (plain gcc, no CUDA).

    ``-ffp-contract=off`` keeps every f32 operation separately rounded, as the
    source is written, on both x86-64 and aarch64.
    """
    with open(_SRC, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()
    stamp = _LIB_PATH + ".sha256"
    if not force and os.path.exists(_LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(
        ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
         "-Wall", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    with open(stamp, "w") as f:
        f.write(digest + "\n")
    return _LIB_PATH


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_q", ctypes.c_int), ("n_kv", ctypes.c_int),
                ("n_iq", ctypes.c_int), ("n_ik", ctypes.c_int), ("weight_fmt", ctypes.c_int),
                ("cache_fmt", ctypes.c_int), ("block_size", ctypes.c_int),
                ("kv_page_stride", ctypes.c_int), ("static_kv_scale", ctypes.c_int),
                ("eps", ctypes.c_float)]


class Caches(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("index_cache", ctypes.c_void_p), ("num_pages16", ctypes.c_int64),
                ("num_index_slots", ctypes.c_int64), ("kv_cache", ctypes.c_void_p),
                ("kv_pages", ctypes.c_int64), ("kv_page_bytes", ctypes.c_int64),
                ("idx_cache", ctypes.c_void_p), ("idx_pages", ctypes.c_int64),
                ("idx_page_bytes", ctypes.c_int64), ("k_global", ctypes.c_float),
                ("v_global", ctypes.c_float)]


class Outputs(ctypes.Structure):
    _fields_ = [("residual", ctypes.c_void_p), ("q_bf16", ctypes.c_void_p),
                ("q_fp8", ctypes.c_void_p), ("iq_bf16", ctypes.c_void_p),
                ("iq_fp8", ctypes.c_void_p), ("q_fp8_scale", ctypes.c_float)]


class DattnConfig(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int), ("q_len", ctypes.c_int), ("bt_width", ctypes.c_int),
                ("window", ctypes.c_int), ("max_blocks", ctypes.c_int), ("part_blocks", ctypes.c_int),
                ("sm_scale", ctypes.c_double)]


class HeadParams(ctypes.Structure):
    _fields_ = [("g_q", ctypes.c_void_p), ("g_k", ctypes.c_void_p), ("g_iq", ctypes.c_void_p),
                ("g_ik", ctypes.c_void_p), ("cos_sin", ctypes.c_void_p),
                ("max_pos", ctypes.c_int64)]


class Inputs(ctypes.Structure):
    _fields_ = [("ar", ctypes.c_void_p), ("res", ctypes.c_void_p), ("g_in", ctypes.c_void_p),
                ("w", ctypes.c_void_p), ("w_scale", ctypes.c_void_p), ("wsf", ctypes.c_void_p),
                ("positions", ctypes.c_void_p), ("slot_mapping", ctypes.c_void_p),
                ("index_slot_mapping", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            f, u8, u16, i64, vp = ctypes.c_float, ctypes.c_uint8, ctypes.c_uint16, ctypes.c_int64, ctypes.c_void_p
            sig = {
                "ora_bf16_decode": (f, [u16]), "ora_bf16_encode": (u16, [f]),
                "ora_e4m3_decode": (f, [u8]), "ora_e4m3_encode": (u8, [f]),
                "ora_e2m1_decode": (f, [u8]), "ora_e2m1_encode": (u8, [f]),
                "ora_e8m0_decode": (ctypes.c_double, [u8]),
                "ora_fp8_scale": (f, [f]), "ora_mx_exponent": (ctypes.c_int, [f]),
                "ora_nvfp4_group16": (None, [vp, ctypes.c_int, f, vp, vp]),
                "ora_page16_of": (i64, [i64, ctypes.c_int]),
                "ora_fp8_k_offset": (i64, [i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
                "ora_fp8_v_offset": (i64, [i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
                "ora_fp8_scale_index": (i64, [i64, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
                "ora_nvfp4_data_offset": (i64, [ctypes.c_int] * 4),
                "ora_nvfp4_sf_linear_offset": (i64, [ctypes.c_int] * 4),
                "ora_nvfp4_sf_vswz_offset": (i64, [ctypes.c_int] * 4),
                "ora_sf128x4_offset": (i64, [i64, i64, i64]),
                "ora_pack_sf128x4": (None, [vp, i64, i64, vp, u8]),
                "ora_head_rmsnorm": (None, [vp, vp, f, vp]),
                "ora_rope_neox": (None, [vp, vp]),
                "ora_prologue_row": (ctypes.c_int, [vp] * 8),
                "ora_project_row": (None, [vp, vp, f, vp, vp, vp, vp, vp]),
                "ora_pre_attn_rows": (ctypes.c_int, [vp, vp, vp, vp, vp, i64, i64, vp, vp, vp, vp]),
                "ora_index_scale_log2e": (ctypes.c_double, [ctypes.c_double]),
                "ora_index_scores": (ctypes.c_int, [vp, i64, vp, i64, vp, ctypes.c_int, vp, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, f, vp, i64]),
                "ora_drafter_qkv": (ctypes.c_int, [vp, i64, i64, vp, vp, f, vp, i64, vp, vp, vp, i64, vp]),
                "ora_drafter_window": (None, [i64, i64, ctypes.c_int, ctypes.c_int, vp, vp]),
                "ora_drafter_attention": (ctypes.c_int, [vp, vp, vp, i64, vp, vp, vp, vp, vp, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def e4m3_encode(x: float) -> int:
    return lib().ora_e4m3_encode(float(x))


def e4m3_decode(c: int) -> float:
    return lib().ora_e4m3_decode(int(c))


def e2m1_encode(x: float) -> int:
    return lib().ora_e2m1_encode(float(x))


def e2m1_decode(c: int) -> float:
    return lib().ora_e2m1_decode(int(c))


def bf16_encode(x: float) -> int:
    return lib().ora_bf16_encode(float(x))


def bf16_decode(b: int) -> float:
    return lib().ora_bf16_decode(int(b))


def e8m0_decode(c: int) -> float:
    return lib().ora_e8m0_decode(int(c))


def mx_exponent(amax: float) -> int:
    return lib().ora_mx_exponent(float(amax))


def fp8_scale(amax: float) -> float:
    return lib().ora_fp8_scale(float(amax))


def nvfp4_group16(v, global_inv: float | None):
    v = np.ascontiguousarray(v, dtype=np.float32)
    assert v.shape == (16,)
    nib = np.zeros(16, np.uint8)
    sf = np.zeros(1, np.uint8)
    lib().ora_nvfp4_group16(_p(v), 0 if global_inv is None else 1,
                            1.0 if global_inv is None else float(global_inv), _p(nib), _p(sf))
    return nib, int(sf[0])


def head_rmsnorm(y, gamma_bf16, eps: float):
    y = np.ascontiguousarray(y, np.float32)
    g = np.ascontiguousarray(gamma_bf16, np.uint16)
    z = np.zeros(HEAD_DIM, np.float64)
    lib().ora_head_rmsnorm(_p(y), _p(g), float(eps), _p(z))
    return z


def rope_neox(z, cs_row_bf16):
    z = np.array(z, np.float64, copy=True)
    cs = np.ascontiguousarray(cs_row_bf16, np.uint16)
    lib().ora_rope_neox(_p(z), _p(cs))
    return z


def pack_sf128x4(src, pad: int = 127):
    """Row-major [R, Ksf] E8M0 codes -> the F8_128x4 layout, R padded to 128."""
    src = np.ascontiguousarray(src, np.uint8)
    R, ksf = src.shape
    rpad = (R + 127) // 128 * 128
    dst = np.zeros(rpad * ksf, np.uint8)
    lib().ora_pack_sf128x4(_p(src), R, ksf, _p(dst), pad)
    return dst


def prologue_row(cfg: Config, ar_row, res_row, g_in):
    H = cfg.hidden
    residual = np.zeros(H, np.uint16)
    xq = np.zeros(H, np.uint8)
    xs = np.zeros(1, np.float32)
    xsf = np.zeros(H // 32, np.uint8)
    rc = lib().ora_prologue_row(ctypes.byref(cfg), _p(np.ascontiguousarray(ar_row, np.uint16)),
                                _p(np.ascontiguousarray(res_row, np.uint16)),
                                _p(np.ascontiguousarray(g_in, np.uint16)),
                                _p(residual), _p(xq), _p(xs), _p(xsf))
    assert rc == 0
    return residual, xq, float(xs[0]), xsf


def project_row(cfg: Config, xq, x_scale, xsf, w, w_scale, wsf):
    N = (cfg.n_q + 2 * cfg.n_kv + cfg.n_iq + cfg.n_ik) * HEAD_DIM
    y = np.zeros(N, np.float32)
    lib().ora_project_row(ctypes.byref(cfg), _p(np.ascontiguousarray(xq, np.uint8)), float(x_scale),
                          _p(None if xsf is None else np.ascontiguousarray(xsf, np.uint8)),
                          _p(np.ascontiguousarray(w, np.uint8)),
                          _p(None if w_scale is None else np.ascontiguousarray(w_scale, np.float32)),
                          _p(None if wsf is None else np.ascontiguousarray(wsf, np.uint8)), _p(y))
    return y


class OracleError(RuntimeError):
    pass


def index_scale_log2e(sm_scale: float) -> float:
    return lib().ora_index_scale_log2e(float(sm_scale))


def index_scores(iq, index_cache, block_table, seq_lens, q_len: int, init_blocks: int, local_blocks: int,
                 index_scale: float, score_cols: int, rows=None, threads: int | None = None):
    """The indexer scores (see ora_index_scores) of a step's rows.

    iq: [M, >=128] bf16 bits (row stride = its second dim); index_cache:
    [slots, 128] E4M3 codes; block_table: [R, bt_width] int32 page-128 block
    ids; seq_lens: [R] int32.  Returns [M, score_cols] float32 with NaN in
    every column the step does not write.  Requests run concurrently on
    `threads` host threads (they are independent); `rows` restricts the
    work to the requests holding those rows."""
    iq = np.ascontiguousarray(iq, np.uint16)
    cache = np.ascontiguousarray(index_cache, np.uint8).reshape(-1)
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    R, bt_width = bt.shape
    M = R * q_len
    assert iq.shape[0] >= M
    out = np.full((M, score_cols), np.nan, np.float32)
    reqs = sorted(set(range(R)) if rows is None else {int(m) // q_len for m in rows})
    L = lib()

    def work(r):
        rc = L.ora_index_scores(_p(iq[r * q_len:]), iq.shape[1], _p(cache), cache.size // HEAD_DIM,
                                _p(bt[r:]), bt_width, _p(sl[r:]), 1, q_len, init_blocks, local_blocks,
                                float(index_scale), _p(out[r * q_len:]), score_cols)
        return rc

    nthreads = threads or min(max(1, len(reqs)), os.cpu_count() or 1)
    if nthreads <= 1:
        rcs = [work(r) for r in reqs]
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            rcs = list(ex.map(work, reqs))
    bad = [rc for rc in rcs if rc != 0]
    if bad:
        raise OracleError(f"oracle index scores returned {bad[0]}")
    return out


def drafter_qkv(qkv, qn, kn, eps: float, cos_sin, positions, slot_mapping, cache):
    """The drafter's q / k head norms, RoPE and FP8 (see ora_drafter_qkv).

    qkv: [M, >=18*128] bf16 bits; qn, kn: [128] bf16 bits; cos_sin:
    [max_pos, 64] bf16 bits; positions, slot_mapping: [M] int64; cache:
    [blocks, 128, 256] uint8, updated in place.  Returns q8 [M * 16, 128]
    E4M3 codes."""
    qkv = np.ascontiguousarray(qkv, np.uint16)
    M = qkv.shape[0]
    q8 = np.zeros((M * 16, HEAD_DIM), np.uint8)
    assert cache.flags.c_contiguous and cache.dtype == np.uint8
    rc = lib().ora_drafter_qkv(_p(qkv), qkv.shape[1], M, _p(np.ascontiguousarray(qn, np.uint16)),
                               _p(np.ascontiguousarray(kn, np.uint16)), float(eps),
                               _p(np.ascontiguousarray(cos_sin, np.uint16)), cos_sin.shape[0],
                               _p(np.ascontiguousarray(positions, np.int64)),
                               _p(np.ascontiguousarray(slot_mapping, np.int64)), _p(cache),
                               cache.size // (128 * 256), _p(q8))
    if rc != 0:
        raise OracleError(f"oracle drafter qkv returned {rc}")
    return q8


def drafter_window(p0: int, seq_len: int, window: int, max_blocks: int):
    lo, hi = ctypes.c_int64(), ctypes.c_int64()
    lib().ora_drafter_window(p0, seq_len, window, max_blocks, ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def drafter_attention(q8, cache, block_table, seq_lens, positions, q_len: int, window: int, max_blocks: int,
                      part_blocks: int, sm_scale: float, rows=None, threads: int | None = None):
    """The drafter's split-KV attention and MXFP8 merge (see
    ora_drafter_attention).  q8: [M * 16, 128] E4M3; cache: [blocks, 128, 256]
    uint8; block_table [R, bt_width] int32; seq_lens [R] int32; positions [M]
    int64.  Returns (out_bf16 [M, 2048] uint16 bits, codes [M, 2048] uint8,
    scales [M, 64] uint8); rows of requests outside `rows` (when given) are
    left zero.  Requests run concurrently on `threads` host threads."""
    q8 = np.ascontiguousarray(q8, np.uint8)
    cache = np.ascontiguousarray(cache, np.uint8)
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    pos = np.ascontiguousarray(positions, np.int64)
    R, bt_width = bt.shape
    M = R * q_len
    assert q8.shape[0] >= M * 16 and pos.shape[0] >= M
    out = np.zeros((M, 2048), np.uint16)
    codes = np.zeros((M, 2048), np.uint8)
    scales = np.zeros((M, 64), np.uint8)
    reqs = sorted(set(range(R)) if rows is None else {int(m) // q_len for m in rows})
    L = lib()
    nblocks = cache.size // (128 * 256)

    def work(r):
        cfg = DattnConfig(1, q_len, bt_width, window, max_blocks, part_blocks, float(sm_scale))
        a = r * q_len
        return L.ora_drafter_attention(ctypes.byref(cfg), _p(q8[a * 16:]), _p(cache), nblocks, _p(bt[r:]),
                                       _p(sl[r:]), _p(pos[a:]), _p(out[a:]), _p(codes[a:]), _p(scales[a:]))

    nthreads = threads or min(max(1, len(reqs)), os.cpu_count() or 1)
    if nthreads <= 1:
        rcs = [work(r) for r in reqs]
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            rcs = list(ex.map(work, reqs))
    bad = [rc for rc in rcs if rc != 0]
    if bad:
        raise OracleError(f"oracle drafter attention returned {bad[0]}")
    return out, codes, scales


def run_rows(wl, state, rows, want_y: bool = False, threads: int | None = None):
    """Run the step for ``rows`` (an iterable of row indices) of workload ``wl``.

    ``state`` is a dict of numpy arrays (see ``workloads.host_state``) whose
    cache and output arrays are updated in place.  Rows are independent, so
    row chunks run concurrently on ``threads`` host threads (ctypes releases
    the GIL); this changes no result.  Returns y [M, N] f32 when ``want_y``.
    """
    L = lib()
    cfg = oracle_config(wl)
    M, N = wl.M, wl.N
    y = np.zeros((M, N), np.float32) if want_y else None
    ins = Inputs(_p(state["ar"]), _p(state["res"]), _p(state["g_in"]), _p(state["w"]),
                 _p(state.get("w_scale")), _p(state.get("wsf")), _p(state["positions"]),
                 _p(state["slot_mapping"]), _p(state.get("index_slot_mapping")))
    hp = HeadParams(_p(state["g_q"]), _p(state["g_k"]), _p(state["g_iq"]), _p(state["g_ik"]),
                    _p(state["cos_sin"]), state["cos_sin"].shape[0])
    cc = Caches()
    if wl.cache_fmt == "fp8":
        cc.k_cache, cc.v_cache = _p(state["k_cache"]), _p(state["v_cache"])
        cc.k_scale, cc.v_scale = _p(state["k_scale"]), _p(state["v_scale"])
        cc.index_cache = _p(state["index_cache"])
        cc.num_pages16 = wl.num_pages16
        cc.num_index_slots = wl.num_index_slots
    else:
        cc.kv_cache, cc.kv_pages, cc.kv_page_bytes = _p(state["kv_cache"]), wl.kv_pages, wl.kv_page_bytes
        cc.idx_cache, cc.idx_pages, cc.idx_page_bytes = _p(state["idx_cache"]), wl.idx_pages, wl.idx_page_bytes
    cc.k_global, cc.v_global = wl.k_global, wl.v_global
    outs = Outputs(_p(state.get("residual")), _p(state.get("q_bf16")), _p(state.get("q_fp8")),
                   _p(state.get("iq_bf16")), _p(state.get("iq_fp8")), wl.q_fp8_scale)
    rows = sorted(set(int(r) for r in rows))
    nthreads = threads or min(max(1, len(rows)), os.cpu_count() or 1)
    per = max(1, -(-len(rows) // (4 * nthreads)))
    # contiguous runs of rows, each cut into pieces of at most `per` rows
    chunks = []
    for r in rows:
        if chunks and chunks[-1][1] == r and chunks[-1][1] - chunks[-1][0] < per:
            chunks[-1][1] = r + 1
        else:
            chunks.append([r, r + 1])

    def work(ab):
        a, b = ab
        return L.ora_pre_attn_rows(ctypes.byref(cfg), ctypes.byref(ins), ctypes.byref(hp),
                                   ctypes.byref(cc), ctypes.byref(outs), a, b, _p(y), None, None, None)

    if nthreads <= 1:
        rcs = [work(c) for c in chunks]
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            rcs = list(ex.map(work, chunks))
    bad = [rc for rc in rcs if rc != 0]
    if bad:
        raise OracleError(f"oracle returned {bad[0]}")
    return y


def oracle_config(wl) -> Config:
    return Config(wl.H, wl.n_q, wl.nkv, wl.n_iq, 1, 0 if wl.weight_fmt == "ptpc" else 1,
                  0 if wl.cache_fmt == "fp8" else 1, wl.block_size, wl.kv_page_stride,
                  1 if wl.static_kv_scale else 0, wl.eps)
