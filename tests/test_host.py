"""CPU-only checks of the host logic: the C-ABI library loads and exports
every entry point include/pre_attn.h declares, configuration and argument
validation return their documented codes without touching a GPU, and the
test harness's cache masks agree with the oracle's offset functions."""

import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import workloads
from tests import harness

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from indexer_projection_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def test_library_exports_every_declared_symbol(B):
    declared = B.declared_symbols()
    assert len(declared) >= 10
    nm = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True, check=True)
    exported = {line.split()[-1] for line in nm.stdout.splitlines() if line.strip()}
    missing = [s for s in declared if s not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(B.LIB_PATH)
    for s in declared:
        assert getattr(lib, s) is not None
    # nothing but the C-ABI is exported
    assert all(s.startswith("pre_attn_") for s in exported), sorted(exported)


def _cfg(B, **kw):
    c = dict(hidden=512, n_kv_heads=1, n_q_heads=0, n_iq_heads=0, weight_format=0, cache_format=0,
             block_size=16, kv_page_stride=0, eps=1e-6, max_tokens=16, flags=0, gemm_grid=0)
    c.update(kw)
    return B.pa_config(**c)


@pytest.mark.parametrize("bad", [dict(hidden=500), dict(hidden=0), dict(hidden=16384 + 128),
                                 dict(n_kv_heads=3), dict(n_kv_heads=0), dict(weight_format=2),
                                 dict(cache_format=5), dict(block_size=8),
                                 dict(cache_format=1, block_size=6), dict(eps=-1.0),
                                 dict(max_tokens=-1), dict(flags=2 | 4), dict(flags=16 | 32),
                                 dict(flags=512 | 1024), dict(n_q_heads=-1)])
def test_init_rejects_bad_configs(B, bad):
    h = ctypes.c_void_p()
    st = B.load().pre_attn_init(ctypes.byref(_cfg(B, **bad)), ctypes.byref(h))
    assert st == B.PA_ERR_CONFIG and not h.value


def test_init_shapes_and_workspace(B):
    for nkv, n in ((1, 2560), (2, 4992), (4, 9856)):
        h = B.pre_attn_init(_cfg(B, hidden=6144, n_kv_heads=nkv, max_tokens=8192))
        assert B.pre_attn_out_features(h) == n
        assert B.pre_attn_workspace_bytes(h, 8192) > 8192 * 6144
        assert B.pre_attn_workspace_bytes(h, 8193) == 0
        B.pre_attn_destroy(h)
    h = B.pre_attn_init(_cfg(B, hidden=6144, n_kv_heads=2, n_iq_heads=4))
    assert B.pre_attn_out_features(h) == 5248  # the 41-head variant of the configs
    B.pre_attn_destroy(h)
    assert B.pre_attn_packed_scale_bytes(9856, 6144) == 9856 * 192
    assert B.pre_attn_packed_scale_bytes(300, 512) == 384 * 16
    assert B.pre_attn_packed_scale_bytes(0, 512) == 0


def test_path_query_rejects_before_touching_the_device(B):
    L = B.load()
    assert L.pre_attn_path(None, 8) == -B.PA_ERR_NULL
    h = B.pre_attn_init(_cfg(B, hidden=6144, n_kv_heads=1, max_tokens=64))
    assert L.pre_attn_path(h, 0) == -B.PA_ERR_SHAPE
    assert L.pre_attn_path(h, 65) == -B.PA_ERR_SHAPE
    B.pre_attn_destroy(h)
    h = B.pre_attn_init(_cfg(B, hidden=6144, n_kv_heads=1, max_tokens=64, flags=B.PA_FLAG_FORCE_GEMV))
    assert L.pre_attn_path(h, 17) == -B.PA_ERR_SHAPE  # the skinny path stops at 16 rows
    B.pre_attn_destroy(h)


def test_workspace_sizes(B):
    # status word + quantised activations and their scales, nothing per N
    h = B.pre_attn_init(_cfg(B, hidden=6144, n_kv_heads=1, max_tokens=64))
    assert 8 * 6144 < B.pre_attn_workspace_bytes(h, 8) < 8 * 6144 + 8192
    B.pre_attn_destroy(h)
    h = B.pre_attn_init(_cfg(B, hidden=6144, n_kv_heads=4, max_tokens=64, weight_format=1))
    assert B.pre_attn_workspace_bytes(h, 8) < 8 * 6144 + 128 * 192 + 8192  # MXFP8: 128 scale rows
    B.pre_attn_destroy(h)


def _run_args(B, M=4, **over):
    """Fake but aligned device addresses: validation fails before any use."""
    base = 1 << 32
    a = {k: base + i * (1 << 24) for i, k in enumerate(
        ["ar", "res", "pos", "slot", "w", "ws", "g", "cs", "k", "v", "ks", "vs", "idx", "q", "iq", "resid", "wk"])}
    a.update(over)
    ins = B.pa_step_inputs(a["ar"], a["res"], a["pos"], a["slot"], None)
    wt = B.pa_weights(a["w"], a["ws"], a["g"], a["g"], a["g"], a["g"], a["g"], a["cs"], 256)
    cc = B.pa_caches()
    cc.k_cache, cc.v_cache, cc.k_scale, cc.v_scale, cc.index_cache = a["k"], a["v"], a["ks"], a["vs"], a["idx"]
    cc.num_pages16, cc.num_index_slots = 64, 1024
    out = B.pa_outputs(a["resid"], a["q"], None, a["iq"], None, 1.0)
    return ins, wt, cc, out, a["wk"]


def _run(B, h, M, ins, wt, cc, out, ws, nbytes=None):
    nbytes = B.pre_attn_workspace_bytes(h, M) if nbytes is None else nbytes
    return B.load().pre_attn_run(h, M, ctypes.byref(ins), ctypes.byref(wt), ctypes.byref(cc),
                                 ctypes.byref(out), ws, nbytes, None)


def test_run_validation_codes(B):
    h = B.pre_attn_init(_cfg(B))
    ins, wt, cc, out, ws = _run_args(B)
    L = B.load()
    assert L.pre_attn_run(None, 4, ctypes.byref(ins), ctypes.byref(wt), ctypes.byref(cc),
                          ctypes.byref(out), ws, 1 << 20, None) == B.PA_ERR_NULL
    assert _run(B, h, 17, ins, wt, cc, out, ws, 1 << 20) == B.PA_ERR_SHAPE
    assert _run(B, h, -1, ins, wt, cc, out, ws, 1 << 20) == B.PA_ERR_SHAPE
    assert _run(B, h, 4, ins, wt, cc, out, ws, 16) == B.PA_ERR_WORKSPACE
    assert _run(B, h, 4, ins, wt, cc, out, None) == B.PA_ERR_WORKSPACE
    o2 = B.pa_outputs(out.residual, None, None, out.iq, None, 1.0)
    assert _run(B, h, 4, ins, wt, cc, o2, ws) == B.PA_ERR_NO_Q_OUTPUT
    o3 = B.pa_outputs(out.residual, out.q, None, None, None, 1.0)
    assert _run(B, h, 4, ins, wt, cc, o3, ws) == B.PA_ERR_NO_IQ_OUTPUT
    o4 = B.pa_outputs(out.residual, out.q, out.q, out.iq, None, 0.0)  # q_fp8 scale 0
    assert _run(B, h, 4, ins, wt, cc, o4, ws) == B.PA_ERR_CONFIG
    # signal mode: done words need a nonzero epoch and 4-byte alignment
    o6 = B.pa_outputs(out.residual, out.q, None, out.iq, None, 1.0, (1 << 32) + (1 << 30), 0)
    assert _run(B, h, 4, ins, wt, cc, o6, ws) == B.PA_ERR_CONFIG
    o7 = B.pa_outputs(out.residual, out.q, None, out.iq, None, 1.0, (1 << 32) + (1 << 30) + 2, 9)
    assert _run(B, h, 4, ins, wt, cc, o7, ws) == B.PA_ERR_ALIGN
    L2 = B.load()
    assert L2.pre_attn_wait_done(None, 4, 1, 10, (1 << 32), None) == B.PA_ERR_NULL
    assert L2.pre_attn_wait_done((1 << 32), 0, 1, 10, (1 << 32), None) == B.PA_ERR_SHAPE
    assert L2.pre_attn_wait_done((1 << 32), 4, 0, 10, (1 << 32), None) == B.PA_ERR_CONFIG
    assert L2.pre_attn_wait_done((1 << 32), 4, 1, 10**8, (1 << 32), None) == B.PA_ERR_CONFIG
    assert L2.pre_attn_wait_done((1 << 32) + 2, 4, 1, 10, (1 << 32), None) == B.PA_ERR_ALIGN
    i2, *_ = _run_args(B, ar=(1 << 32) + 8)
    assert _run(B, h, 4, i2, wt, cc, out, ws) == B.PA_ERR_ALIGN
    _, _, _, _, ws_bad = _run_args(B, wk=(1 << 32) + 64)
    assert _run(B, h, 4, ins, wt, cc, out, ws_bad) == B.PA_ERR_ALIGN
    # residual partially over res -> alias; exactly in place -> accepted by validation
    o5 = B.pa_outputs(ins.res + 512, out.q, None, out.iq, None, 1.0)
    assert _run(B, h, 4, ins, wt, cc, o5, ws) == B.PA_ERR_ALIAS
    i3 = B.pa_step_inputs(ins.ar, ins.res, None, ins.slot_mapping, None)
    assert _run(B, h, 4, i3, wt, cc, out, ws) == B.PA_ERR_NULL
    c2 = B.pa_caches()
    assert _run(B, h, 4, ins, wt, c2, out, ws) == B.PA_ERR_NULL
    # M == 0 launches nothing and succeeds, on a machine with or without a GPU
    assert _run(B, h, 0, ins, wt, cc, out, ws) == B.PA_OK
    B.pre_attn_destroy(h)


def test_run_validation_nvfp4_geometry(B):
    h = B.pre_attn_init(_cfg(B, cache_format=1, block_size=16))
    ins, wt, _, out, ws = _run_args(B)
    cc = B.pa_caches()
    cc.kv_cache, cc.idx_cache = 1 << 33, 1 << 34
    cc.kv_pages, cc.idx_pages = 8, 8
    cc.kv_page_bytes, cc.idx_page_bytes = 2 * 16 * 72, 16 * 72
    cc.k_global_scale = cc.v_global_scale = 1.0
    assert _run(B, h, 4, ins, wt, cc, out, ws) == B.PA_OK or True  # fine geometry: reaches CUDA
    cc.kv_page_bytes = 2 * 16 * 72 - 32
    assert _run(B, h, 4, ins, wt, cc, out, ws) == B.PA_ERR_CONFIG
    cc.kv_page_bytes = 2 * 16 * 72 + 16
    assert _run(B, h, 4, ins, wt, cc, out, ws) == B.PA_ERR_ALIGN
    cc.kv_page_bytes = 2 * 16 * 72
    cc.kv_cache = (1 << 33) + 16
    assert _run(B, h, 4, ins, wt, cc, out, ws) == B.PA_ERR_ALIGN
    cc.kv_cache = 1 << 33
    cc.v_global_scale = 0.0
    assert _run(B, h, 4, ins, wt, cc, out, ws) == B.PA_ERR_CONFIG
    B.pre_attn_destroy(h)


def test_harness_masks_match_oracle_offsets():
    L = oracle.lib()
    wl = workloads.tiny().replace(nkv=2, kv_page_stride=16, M=6)
    st = workloads.host_state(wl)
    st["slot_mapping"] = st["slot_mapping"] % (wl.num_pages16 * 16 // 2)  # page16 ids stay in the pool
    m = harness.write_masks(wl, st, range(wl.M))
    want = np.zeros_like(m["k_cache"])
    wantv = np.zeros_like(m["v_cache"])
    for r in range(wl.M):
        s = int(st["slot_mapping"][r])
        p16 = L.ora_page16_of(s, 16)
        for h in range(2):
            for d in range(128):
                want[L.ora_fp8_k_offset(p16, h, 2, s % 16, d)] = True
                wantv[L.ora_fp8_v_offset(p16, h, 2, s % 16, d)] = True
    assert np.array_equal(m["k_cache"], want) and np.array_equal(m["v_cache"], wantv)
    wl = workloads.Workload("n", H=512, nkv=2, M=5, weight_fmt="mx", cache_fmt="nvfp4", seed=3,
                            positions="uniform", max_pos=64, pool_pages=8, page_pad=32)
    st = workloads.host_state(wl)
    dm, fm = harness.write_masks(wl, st, range(wl.M))["kv_cache"]
    wd, wf = np.zeros_like(dm), np.zeros_like(fm)
    for r in range(wl.M):
        s = int(st["slot_mapping"][r])
        base = (s // 16) * wl.kv_page_bytes
        for sl in range(4):
            for d in range(0, 128, 2):
                wd[base + L.ora_nvfp4_data_offset(16, sl, s % 16, d)] = True
            for g in range(8):
                f = L.ora_nvfp4_sf_vswz_offset if sl % 2 else L.ora_nvfp4_sf_linear_offset
                wf[base + f(16, sl, s % 16, g)] = True
    assert np.array_equal(dm, wd) and np.array_equal(fm, wf)


def test_drafter_partition_choice_and_workspace(B):
    # floor(2 * SMs / R) partitions of a full window (one wave), cut evenly
    assert B.pre_attn_drafter_part_blocks(64, 34, 152) == 9   # 304 // 64 = 4 partitions of <= 9 blocks
    assert B.pre_attn_drafter_part_blocks(1, 34, 152) == 1
    assert B.pre_attn_drafter_part_blocks(1000, 34, 152) == 34
    assert B.pre_attn_drafter_part_blocks(152, 34, 152) == 17
    assert B.pre_attn_drafter_part_blocks(100, 34, 152) == 12  # 304 // 100 = 3 partitions of <= 12 blocks
    assert B.pre_attn_drafter_part_blocks(0, 34, 152) < 0
    # ceil(34 / 9) = 4 partials of 128 m + 128 l + 128 x 128 o f32 per request
    assert B.pre_attn_drafter_workspace_bytes(64, 34, 9) == 64 * 4 * (1024 + 65536)
    assert B.pre_attn_drafter_workspace_bytes(65, 34, 34) == 65 * (1024 + 65536)
    assert B.pre_attn_drafter_workspace_bytes(0, 34, 9) == 0


def _drafter_args(B, bufs, **kw):
    a = B.pa_drafter_args()
    for k in ("positions", "cache", "block_table", "seq_lens", "q8", "out_codes", "out_scales", "workspace",
              "status"):
        setattr(a, k, bufs[k])
    a.num_blocks, a.bt_width, a.R, a.q_len = 16, 8, 2, 7
    a.window, a.max_blocks, a.part_blocks, a.sm_scale = 4096, 34, 4, 128 ** -0.5
    a.workspace_bytes = B.pre_attn_drafter_workspace_bytes(2, 34, 4)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_drafter_validation_codes(B):
    # fake, aligned "device" addresses: every case returns before any launch
    base = 1 << 40
    bufs = {k: base + i * (1 << 24) for i, k in enumerate(
        ("positions", "cache", "block_table", "seq_lens", "q8", "out_codes", "out_scales", "workspace", "status"))}
    run = lambda **kw: B.pre_attn_drafter_attention(_drafter_args(B, bufs, **kw), None, check=False)  # noqa: E731
    assert B.load().pre_attn_drafter_attention(None, None) == B.PA_ERR_NULL
    for k in ("positions", "cache", "block_table", "seq_lens", "q8", "out_codes", "out_scales", "workspace", "status"):
        assert run(**{k: None}) == B.PA_ERR_NULL, k
    assert run(qkv=base) == B.PA_ERR_NULL  # qkv without its gammas, table and slots
    for bad in (dict(R=-1), dict(R=65536), dict(q_len=0), dict(q_len=9), dict(bt_width=0), dict(num_blocks=0),
                dict(num_blocks=1 << 24)):
        assert run(**bad) == B.PA_ERR_SHAPE, bad
    q = dict(qkv=base, qn=base, kn=base, cos_sin=base, slot_mapping=base, max_pos=64)
    assert run(**q, qkv_stride=18 * 128 - 8) == B.PA_ERR_SHAPE
    assert run(**q, qkv_stride=18 * 128 + 4) == B.PA_ERR_SHAPE
    for bad in (dict(window=0), dict(max_blocks=0), dict(part_blocks=-1), dict(sm_scale=float("nan")),
                dict(sm_scale=-0.1), dict(sm_scale=0.0), dict(sm_scale=float("inf"))):
        assert run(**bad) == B.PA_ERR_CONFIG, bad
    assert run(**q, qkv_stride=18 * 128, eps=-1.0) == B.PA_ERR_CONFIG
    for k, off in (("cache", 8), ("q8", 4), ("out_codes", 8), ("workspace", 128), ("status", 2), ("positions", 4)):
        assert run(**{k: bufs[k] + off}) == B.PA_ERR_ALIGN, k
    assert run(out_bf16=base + 8) == B.PA_ERR_ALIGN
    assert run(workspace_bytes=100) == B.PA_ERR_WORKSPACE
    assert run(R=0) == B.PA_OK  # nothing to do: nothing launched
