"""Shared test machinery: device buffers for a workload, the CUDA run through
the C-ABI, the oracle run, and the comparison at the tolerances of the step.

Tolerances (the step's contract):
  * residual: bit-exact (bf16(ar + res) with an f32 add on both sides);
  * bf16 outputs: |gpu - oracle| <= 1e-2 + 2e-2 |oracle|;
  * FP8 / NVFP4 codes (outputs, cache data and NVFP4 scale bytes): at most one
    code step apart (+0 and -0 equal) in at most 0.1% of the elements;
  * f32 per-token cache scales: relative 1e-3;
  * cache bytes no row should write: untouched (sentinel) bit-exactly, and the
    written (page, token, byte) set equal to the oracle's.
"""

from __future__ import annotations

import numpy as np

import oracle
import workloads
from workloads import HEAD_DIM, SENTINEL

BF16_ATOL, BF16_RTOL = 1e-2, 2e-2
CODE_FRAC = 1e-3
SCALE_RTOL = 1e-3

# ------------------------------------------------------------- code helpers

def bf16_to_f32(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)


def e4m3_ordinal(c):
    c = np.asarray(c, np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def e2m1_ordinal(n):
    n = np.asarray(n, np.int32)
    mag = n & 7
    return np.where(n & 8, -mag, mag)


class CodeTally:
    """Counts of compared and differing FP8 / NVFP4 codes over one step."""

    def __init__(self):
        self.n = 0
        self.diff = 0
        self.parts = []

    def check(self, frac=CODE_FRAC, tag=""):
        assert self.diff <= frac * self.n, (
            f"{tag} {self.diff}/{self.n} codes differ by one step (> {frac:.1%}): {self.parts}")


def check_codes(gpu, ref, name, ordinal=e4m3_ordinal, tally=None, frac=CODE_FRAC):
    """Every code within one step; the share of differing codes is checked
    per array, or pooled over the step's code outputs when `tally` is given."""
    gpu, ref = np.asarray(gpu).reshape(-1), np.asarray(ref).reshape(-1)
    assert gpu.shape == ref.shape, name
    if gpu.size == 0:
        return
    d = np.abs(ordinal(gpu) - ordinal(ref))
    bad = int((d > 1).sum())
    assert bad == 0, f"{name}: {bad} codes more than one step apart (max {d.max()}), first at {np.argmax(d > 1)}"
    nd = int((d > 0).sum())
    if tally is None:
        assert nd <= frac * d.size, f"{name}: {nd}/{d.size} codes differ (> {frac:.1%})"
    else:
        tally.n += d.size
        tally.diff += nd
        tally.parts.append((name, nd, d.size))


def check_bf16(gpu, ref, name):
    g, o = bf16_to_f32(gpu), bf16_to_f32(ref)
    err = np.abs(g.astype(np.float64) - o) - (BF16_ATOL + BF16_RTOL * np.abs(o))
    assert np.all(err <= 0), f"{name}: max excess {err.max():.3g} at {np.argmax(err)}"


def check_nvfp4_data(gpu, ref, name, tally=None):
    g, o = np.asarray(gpu, np.uint8), np.asarray(ref, np.uint8)
    gn = np.stack([g & 15, g >> 4], -1).reshape(-1)
    on = np.stack([o & 15, o >> 4], -1).reshape(-1)
    check_codes(gn, on, name, ordinal=e2m1_ordinal, tally=tally)


# ---------------------------------------------------------- write masks

def _page16_of(slot, kps):
    slot = np.asarray(slot, np.int64)
    if kps == 8:
        return slot // 16
    return (slot // 128) * kps + (slot % 128) // 16


def write_masks(wl, st, rows):
    """Byte masks of what the step writes for `rows` (numpy formulas of the
    cache layouts; pinned against the oracle's offset functions in
    test_harness_masks_match_oracle_offsets)."""
    rows = np.asarray(sorted(rows), np.int64)
    slots = st["slot_mapping"][rows]
    islots = st["index_slot_mapping"][rows]
    d = np.arange(HEAD_DIM)
    masks = {}
    if wl.cache_fmt == "fp8":
        v = slots >= 0
        s = slots[v]
        p16, t = _page16_of(s, wl.kv_page_stride), s % 16
        km = np.zeros(st["k_cache"].size, bool)
        vm = np.zeros(st["v_cache"].size, bool)
        sm = np.zeros(st["k_scale"].size, bool)
        for h in range(wl.nkv):
            base = (p16 * wl.nkv + h) * 2048
            km[(base[:, None] + (d // 16) * 256 + t[:, None] * 16 + d % 16).reshape(-1)] = True
            vm[(base[:, None] + d * 16 + t[:, None]).reshape(-1)] = True
            sm[(p16 * wl.nkv + h) * 16 + t] = True
        im = np.zeros(st["index_cache"].size, bool)
        iv = islots[islots >= 0]
        im[(iv[:, None] * HEAD_DIM + d).reshape(-1)] = True
        masks.update(k_cache=km, v_cache=vm, k_scale=sm, v_scale=sm.copy(), index_cache=im)
    else:
        bs = wl.block_size

        def nv(cache_size, page_bytes, sl_list, sl_vswz, sv):
            dm = np.zeros(cache_size, bool)
            fm = np.zeros(cache_size, bool)
            page, t = sv // bs, sv % bs
            for sl in sl_list:
                base = page * page_bytes + sl * bs * 72
                dm[(base[:, None] + t[:, None] * 64 + np.arange(64)).reshape(-1)] = True
                g = np.arange(8)
                if sl in sl_vswz:
                    off = ((t[:, None] // 4) * 4 + g // 2) * 8 + (g % 2) * 4 + t[:, None] % 4
                else:
                    off = t[:, None] * 8 + g
                fm[(base[:, None] + bs * 64 + off).reshape(-1)] = True
            return dm, fm

        s = slots[slots >= 0]
        dm, fm = nv(st["kv_cache"].size, wl.kv_page_bytes, range(2 * wl.nkv),
                    set(range(1, 2 * wl.nkv, 2)), s)
        iv = islots[islots >= 0]
        idm, ifm = nv(st["idx_cache"].size, wl.idx_page_bytes, [0], set(), iv)
        masks.update(kv_cache=(dm, fm), idx_cache=(idm, ifm))
    return masks


# ----------------------------------------------------------- comparisons

def compare(wl, gpu, ref, rows, all_rows=None, where=""):
    """Compare GPU results with oracle results on `rows` (oracle ran on
    exactly those rows).  `all_rows`: every row the GPU ran (defaults to
    rows), used to check that nothing outside their slots was written."""
    rows = np.asarray(sorted(rows), np.int64)
    all_rows = rows if all_rows is None else np.asarray(sorted(all_rows), np.int64)
    tag = f"[{wl.name}{where}]"
    tally = CodeTally()
    # outputs
    if "residual" in gpu and gpu["residual"] is not None:
        g, o = gpu["residual"][rows], ref["residual"][rows]
        nbad = int((g != o).sum())
        assert nbad == 0, f"{tag} residual: {nbad} elements differ"
    for k in ("q_bf16", "iq_bf16"):
        if k in ref:
            check_bf16(gpu[k][rows], ref[k][rows], f"{tag} {k}")
    for k in ("q_fp8", "iq_fp8"):
        if k in ref:
            check_codes(gpu[k][rows], ref[k][rows], f"{tag} {k}", tally=tally)
    # caches
    m_rows = write_masks(wl, ref, rows)
    m_all = write_masks(wl, ref, all_rows)
    if wl.cache_fmt == "fp8":
        for k in ("k_cache", "v_cache", "index_cache"):
            g, o = gpu[k], ref[k]
            outside = ~m_all[k]
            assert np.all(g[outside] == SENTINEL), f"{tag} {k}: {int((g[outside] != SENTINEL).sum())} bytes written outside the slots"
            check_codes(g[m_rows[k]], o[m_rows[k]], f"{tag} {k}", tally=tally)
        for k in ("k_scale", "v_scale"):
            g, o = gpu[k], ref[k]
            outside = ~m_all[k]
            assert np.all(g.view(np.uint32)[outside] == 0xA5A5A5A5), f"{tag} {k} written outside the slots"
            gm, om = g[m_rows[k]].astype(np.float64), o[m_rows[k]].astype(np.float64)
            assert np.all(np.abs(gm - om) <= SCALE_RTOL * np.abs(om)), f"{tag} {k}: scales differ"
    else:
        for k in ("kv_cache", "idx_cache"):
            g, o = gpu[k], ref[k]
            dm_r, fm_r = m_rows[k]
            dm_a, fm_a = m_all[k]
            outside = ~(dm_a | fm_a)
            assert np.all(g[outside] == SENTINEL), f"{tag} {k}: {int((g[outside] != SENTINEL).sum())} bytes written outside the slots"
            check_nvfp4_data(g[dm_r], o[dm_r], f"{tag} {k} data", tally=tally)
            check_codes(g[fm_r], o[fm_r], f"{tag} {k} scales", tally=tally)
    tally.check(tag=tag)
    return tally


# ------------------------------------------------------------ GPU side

class GpuRun:
    """Device copies of a workload's state and a configured PreAttn."""

    def __init__(self, wl, st, flags=0, max_tokens=None, gemm_grid=0, device="cuda"):
        import torch

        from indexer_projection_gb300 import binding as B
        from indexer_projection_gb300.runner import PreAttn

        self.torch, self.B = torch, B
        self.wl, self.st = wl, st
        dev = torch.device(device)
        self.dev = dev

        def t(a):
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                a = a.view(np.int16)
            if a.dtype == np.uint32:
                a = a.view(np.int32)
            return torch.from_numpy(a.copy()).to(dev)

        self.t = t
        self.d = {k: t(v) for k, v in st.items() if isinstance(v, np.ndarray)}
        wf = B.PA_WEIGHT_FP8_PER_CHANNEL if wl.weight_fmt == "ptpc" else B.PA_WEIGHT_MXFP8
        cf = B.PA_CACHE_FP8 if wl.cache_fmt == "fp8" else B.PA_CACHE_NVFP4
        self.runner = PreAttn(wl.H, wl.nkv, weight_format=wf, cache_format=cf,
                              max_tokens=max(wl.M, 1) if max_tokens is None else max_tokens,
                              block_size=wl.block_size, eps=wl.eps, n_q_heads=wl.n_q, n_iq_heads=wl.n_iq,
                              kv_page_stride=wl.kv_page_stride,
                              flags=flags | (B.PA_FLAG_STATIC_KV_SCALE if wl.static_kv_scale else 0),
                              gemm_grid=gemm_grid, device=dev)
        if wl.weight_fmt == "mx":
            nb = B.pre_attn_packed_scale_bytes(wl.N, wl.H)
            self.wsf_packed = torch.empty(nb, dtype=torch.uint8, device=dev)
            B.pre_attn_pack_scales(self.d["wsf"], self.wsf_packed, wl.N, wl.H)
            wscale = self.wsf_packed
        else:
            wscale = self.d["w_scale"]
        d = self.d
        self.weights = PreAttn.weights(d["w"], wscale, d["g_in"], d["g_q"], d["g_k"], d["g_iq"], d["g_ik"],
                                       d["cos_sin"])
        if wl.cache_fmt == "fp8":
            self.caches = PreAttn.fp8_caches(d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                                             d["index_cache"], wl.num_pages16, wl.num_index_slots)
        else:
            self.caches = PreAttn.nvfp4_caches(d["kv_cache"], wl.kv_pages, wl.kv_page_bytes, d["idx_cache"],
                                               wl.idx_pages, wl.idx_page_bytes, wl.k_global, wl.v_global)
        self.done = None
        self.set_done_epoch(0)

    def set_done_epoch(self, epoch: int):
        """Ask for the step's done words (signal mode) with this epoch (0: none)."""
        from indexer_projection_gb300.runner import PreAttn

        d, wl = self.d, self.wl
        if epoch and self.done is None:
            self.done = self.torch.zeros(max(wl.M, 1) * wl.n_heads, dtype=self.torch.int32, device=self.dev)
        self.outputs = PreAttn.outputs(d.get("residual"), d.get("q_bf16"), d.get("q_fp8"), d.get("iq_bf16"),
                                       d.get("iq_fp8"), wl.q_fp8_scale, done=self.done if epoch else None,
                                       done_epoch=epoch)

    def run(self, M=None, check=True):
        d = self.d
        return self.runner.run(self.wl.M if M is None else M, d["ar"], d["res"], d["positions"],
                               d["slot_mapping"], self.weights, self.caches, self.outputs,
                               index_slot_mapping=d["index_slot_mapping"], check=check)

    def results(self):
        self.torch.cuda.synchronize()
        out = {}
        for k in workloads.CACHE_KEYS + workloads.OUTPUT_KEYS:
            if k in self.d:
                a = self.d[k].cpu().numpy()
                out[k] = a.view(self.st[k].dtype).reshape(self.st[k].shape)
        return out


def fresh_reference(wl, st):
    """A copy of the state whose outputs and caches are back at the sentinel."""
    ref = dict(st)
    for k in workloads.CACHE_KEYS + workloads.OUTPUT_KEYS:
        if k in st:
            ref[k] = st[k].copy()
    return ref


def oracle_run(wl, st, rows):
    ref = fresh_reference(wl, st)
    oracle.run_rows(wl, ref, rows)
    return ref


def sample_rows(M, n, seed=0, must=()):
    rng = np.random.default_rng(seed)
    base = {0, M - 1, *[r for r in must if 0 <= r < M]}
    for b in (127, 128, 255, 256, 383, 384):
        if b < M:
            base.add(b)
    extra = rng.choice(M, size=min(M, n), replace=False)
    return sorted(base | set(int(x) for x in extra))
