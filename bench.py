#!/usr/bin/env python
"""Benchmark of the MiniMax-M3 pre-attention step on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--workload decode|spec_decode|prefill|tiny|sweep_m<M>]

A step is one pre_attn_run() (prologue + skinny GEMV or tcgen05 GEMM with the
fused head epilogue) over one batch of the workload's synthetic inputs.  The
timed region is a CUDA graph of exactly K steps; step i uses the i-th of C
rotating copies of the layer weights and inputs (C chosen so the copies
exceed twice the L2), so weights stream from HBM as they would across layers.
Rank 0 prints one JSON line.  Under torchrun each rank runs an independent
replica (the step has no cross-GPU exchange) and the slowest rank's time sets
the aggregate tokens/s.

--impl reference times the CPU oracle (tests only use it otherwise) on the
host cores on bounded samples of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "pre-attn µs/layer & tokens/s; % HBM roofline (decode), % FP8 peak (prefill)"
FP8_OVER_BF16 = 4.5 / 2.25  # nominal dense FP8 : BF16 tensor rate on GB300


def get_workload(name: str):
    if name.startswith("sweep_m"):
        return workloads.sweep(int(name[len("sweep_m"):]))
    return workloads.CONFIGS[name]()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------- byte / flop accounting

def step_bytes(wl) -> dict:
    """Algorithmic bytes of one step: every input read once, every output
    written once (workspace scratch excluded)."""
    M, H, N = wl.M, wl.H, wl.N
    w = N * H + (4 * N if wl.weight_fmt == "ptpc" else N * H // 32)
    act_in = 2 * M * H * 2
    resid = M * H * 2
    qb = M * wl.n_q * 128 * ((2 if wl.q_bf16 else 0) + (1 if wl.q_fp8 else 0))
    iqb = M * wl.n_iq * 128 * ((2 if wl.iq_bf16 else 0) + (1 if wl.iq_fp8 else 0))
    if wl.cache_fmt == "fp8":
        cache = M * (wl.nkv * 2 * (128 + 4) + 128)
    else:
        cache = M * (2 * wl.nkv + 1) * 72
    meta = M * 8 * 3 + M * 64 * 2 + 4 * 128 * 2 + H * 2
    xq = M * H + (4 * M if wl.weight_fmt == "ptpc" else M * H // 32)
    main = w + xq + qb + iqb + cache + meta - H * 2  # the main kernel: weights, xq, outputs
    return {"step": w + act_in + resid + qb + iqb + cache + meta, "main": main, "weights": w}


def step_flops(wl) -> int:
    return 2 * wl.M * wl.N * wl.H


KERNEL_SOURCES = {"gemv": ("pa_gemv.cu", "pa_device.cuh", "pa_tc.cuh", "pa_norm.cuh"),
                  "gemv_fused": ("pa_gemv.cu", "pa_device.cuh", "pa_tc.cuh", "pa_norm.cuh"),
                  "gemm": ("pa_gemm.cu", "pa_device.cuh", "pa_tc.cuh"),
                  "gemm2": ("pa_gemm2.cu", "pa_device.cuh"),
                  "prologue": ("pa_prologue.cu", "pa_device.cuh", "pa_norm.cuh")}


def kernel_sha(kernel: str) -> str:
    """Hash of the sources a kernel is built from (ties an ncu summary to them)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "indexer_projection_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.lstrip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_sources_sha256_16") != kernel_sha(kernel):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.period = period_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period), "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0=None, t1=None):
        sel = [p for (t, p) in self.samples if (t0 is None or t >= t0) and (t1 is None or t <= t1)]
        if not sel:
            sel = [p for (_, p) in self.samples]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in sel if num(p[0]) is not None]
        mx = [num(p[1]) for p in sel if num(p[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in sel:
            for name, v in zip(names, p[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sel)}


# ------------------------------------------------------------ several ranks

def max_over_ranks(values, world: int, device=None):
    """Element-wise max of `values` over the ranks (the slowest rank's times);
    the input itself when there is one rank."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def tokens_per_second(world: int, rows_per_step: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own rows each step."""
    return world * rows_per_step / (ms_per_step * 1e-3)


# ----------------------------------------------------------------- our arm

class DeviceWorkload:
    """C rotating copies of a workload's weights and inputs on the device."""

    def __init__(self, wl, st, copies: int, device, flags=0):
        import torch

        from indexer_projection_gb300 import binding as B
        from indexer_projection_gb300.runner import PreAttn

        self.torch, self.B, self.wl = torch, B, wl
        self.dev = device

        def t(a):
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                a = a.view(np.int16)
            return torch.from_numpy(a).to(device)

        wf = B.PA_WEIGHT_FP8_PER_CHANNEL if wl.weight_fmt == "ptpc" else B.PA_WEIGHT_MXFP8
        cf = B.PA_CACHE_FP8 if wl.cache_fmt == "fp8" else B.PA_CACHE_NVFP4
        self.runner = PreAttn(wl.H, wl.nkv, weight_format=wf, cache_format=cf, max_tokens=wl.M,
                              block_size=wl.block_size, eps=wl.eps, n_q_heads=wl.n_q, n_iq_heads=wl.n_iq,
                              kv_page_stride=wl.kv_page_stride, flags=flags, device=device)
        # layer copies: the first is the drawn weight, the rest are byte-rolled
        # variants (same value distribution, different bytes) so no copy hits
        # another's L2 lines
        self.layers = []
        w0 = t(st["w"])
        g = {k: t(st[k]) for k in ("g_in", "g_q", "g_k", "g_iq", "g_ik")}
        cs = t(st["cos_sin"])
        if wl.weight_fmt == "ptpc":
            s0 = t(st["w_scale"])
        else:
            wsf = t(st["wsf"])
            s0 = torch.empty(B.pre_attn_packed_scale_bytes(wl.N, wl.H), dtype=torch.uint8, device=device)
            B.pre_attn_pack_scales(wsf, s0, wl.N, wl.H)
        ar0, res0 = t(st["ar"]), t(st["res"])
        for c in range(copies):
            w = w0 if c == 0 else torch.roll(w0, shifts=c * 7919, dims=1).contiguous()
            ar = ar0 if c == 0 else torch.roll(ar0, shifts=c * 131, dims=1).contiguous()
            res = res0 if c == 0 else torch.roll(res0, shifts=c * 257, dims=1).contiguous()
            s = s0 if c == 0 else s0.clone()
            self.layers.append(dict(w=w, s=s, ar=ar, res=res,
                                    wt=PreAttn.weights(w, s, g["g_in"], g["g_q"], g["g_k"], g["g_iq"], g["g_ik"], cs)))
        self.keep = (g, cs)
        self.pos, self.slot = t(st["positions"]), t(st["slot_mapping"])
        self.islot = t(st["index_slot_mapping"])
        if wl.cache_fmt == "fp8":
            self.cache_t = {k: t(st[k]) for k in ("k_cache", "v_cache", "k_scale", "v_scale", "index_cache")}
            c = self.cache_t
            self.caches = PreAttn.fp8_caches(c["k_cache"], c["v_cache"], c["k_scale"], c["v_scale"],
                                             c["index_cache"], wl.num_pages16, wl.num_index_slots)
        else:
            self.cache_t = {k: t(st[k]) for k in ("kv_cache", "idx_cache")}
            c = self.cache_t
            self.caches = PreAttn.nvfp4_caches(c["kv_cache"], wl.kv_pages, wl.kv_page_bytes, c["idx_cache"],
                                               wl.idx_pages, wl.idx_page_bytes, wl.k_global, wl.v_global)
        M = wl.M
        self.out_t = dict(residual=torch.empty(M, wl.H, dtype=torch.int16, device=device))
        if wl.q_bf16:
            self.out_t["q"] = torch.empty(M, wl.n_q * 128, dtype=torch.int16, device=device)
        if wl.q_fp8:
            self.out_t["q_fp8"] = torch.empty(M, wl.n_q * 128, dtype=torch.uint8, device=device)
        if wl.iq_bf16:
            self.out_t["iq"] = torch.empty(M, wl.n_iq * 128, dtype=torch.int16, device=device)
        if wl.iq_fp8:
            self.out_t["iq_fp8"] = torch.empty(M, wl.n_iq * 128, dtype=torch.uint8, device=device)
        o = self.out_t
        self.outputs = PreAttn.outputs(o.get("residual"), o.get("q"), o.get("q_fp8"), o.get("iq"),
                                       o.get("iq_fp8"), wl.q_fp8_scale)

    def step(self, i: int, stream=None):
        L = self.layers[i % len(self.layers)]
        self.runner.run(self.wl.M, L["ar"], L["res"], self.pos, self.slot, L["wt"], self.caches, self.outputs,
                        index_slot_mapping=self.islot, stream=stream)


def run_ours(args, wl, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from indexer_projection_gb300 import binding as B

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks, peak_src = measured_peaks()
    st = workloads.host_state(wl)
    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    per_copy = step_bytes(wl)["weights"] + 2 * wl.M * wl.H * 2
    copies = max(2, min(64, math.ceil(2.5 * l2 / per_copy)))
    flags = {"auto": 0, "single": B.PA_FLAG_GEMM_SINGLE, "pair": B.PA_FLAG_GEMM_PAIR}[args.gemm]
    if args.fuse:
        flags |= B.PA_FLAG_FUSE
    dw = DeviceWorkload(wl, st, copies, dev, flags=flags)
    stream = torch.cuda.Stream(dev)
    K, W = args.steps, args.warmup

    def barrier():
        if world > 1:
            dist.barrier()

    sampler = ClockSampler(local_rank)
    sampler.start()
    with torch.cuda.stream(stream):
        for i in range(W):
            dw.step(i, stream)
    stream.synchronize()
    # a CUDA graph of exactly K steps (PDL edges kept between the kernels)
    G = min(K, 4096)
    full, rest = divmod(K, G)
    graphs = []
    for n in ([G] if full else []) + ([rest] if rest else []):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                dw.step(i, stream)
        graphs.append((g, n))
    with torch.cuda.stream(stream):
        for g, _ in graphs:  # untimed replay: instantiation / first-launch costs
            g.replay()
    stream.synchronize()
    barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(full):
            graphs[0][0].replay()
        if rest:
            graphs[-1][0].replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier()
    ms = max_over_ranks([e0.elapsed_time(e1)], world, dev)[0]
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    del graphs

    # main-kernel device time: events recorded around it on the launching
    # stream, steps queued behind a GPU sleep long enough that the host never
    # starves the GPU between them (else the events would time the host's
    # launch calls); no programmatic overlap with the prologue here
    P = min(max(K, 50), 400)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(P)]
    for a, b in evs:  # torch creates its CUDA events on first record
        a.record(stream)
        b.record(stream)
    stream.synchronize()

    def profiled_steps(n):
        for i in range(n):
            B.pre_attn_set_profile_events(dw.runner.handle, evs[i][0], evs[i][1])
            dw.step(i, stream)

    with torch.cuda.stream(stream):
        t_h = time.perf_counter()
        profiled_steps(min(P, 20))
        host_s = (time.perf_counter() - t_h) / min(P, 20)  # host time to queue one step
    stream.synchronize()
    sleep_cycles = int(3.0 * P * host_s * 2.1e9)  # three times the queueing time at <= 2.1 GHz
    with torch.cuda.stream(stream):
        torch.cuda._sleep(sleep_cycles)
        profiled_steps(P)
    B.pre_attn_set_profile_events(dw.runner.handle, None, None)
    stream.synchronize()
    main_ms = statistics.median(a.elapsed_time(b) for a, b in evs[P // 4:])

    # end to end through the public API: pinned host inputs in, results out,
    # every step.  The step's inputs sit in one pinned host block and one
    # device block (ar | res | positions | slots, each 256-byte aligned), its
    # outputs in one device block and one pinned host block: one copy each
    # way per step (per-copy overhead, not bytes, dominated nine copies).
    from indexer_projection_gb300.runner import PreAttn
    E = min(K, 2000)
    def layout(arrays):
        offs, off = [], 0
        for a in arrays:
            offs.append(off)
            off = (off + a.numel() * a.element_size() + 255) // 256 * 256
        return offs, off

    def views(block, offs, like):
        return [block[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape) for o, x in zip(offs, like)]

    src_in = [torch.from_numpy(st["ar"].view(np.int16)), torch.from_numpy(st["res"].view(np.int16)),
              torch.from_numpy(st["positions"]), torch.from_numpy(st["slot_mapping"])]
    in_offs, in_bytes = layout(src_in)
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    for v, x in zip(views(h_in, in_offs, src_in), src_in):
        v.copy_(x)
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    d_ar, d_res, d_pos, d_slot = views(d_in, in_offs, src_in)
    out_keys = list(dw.out_t)
    out_like = [dw.out_t[k] for k in out_keys]
    out_offs, out_bytes = layout(out_like)
    d_out = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    d_o = dict(zip(out_keys, views(d_out, out_offs, out_like)))
    e2e_outputs = PreAttn.outputs(d_o.get("residual"), d_o.get("q"), d_o.get("q_fp8"), d_o.get("iq"),
                                  d_o.get("iq_fp8"), wl.q_fp8_scale)
    h_out = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in src_in)
    d2h = sum(x.numel() * x.element_size() for x in out_like)
    def e2e_step(i):
        d_in.copy_(h_in, non_blocking=True)
        Li = dw.layers[i % len(dw.layers)]
        dw.runner.run(wl.M, d_ar, d_res, d_pos, d_slot, Li["wt"], dw.caches, e2e_outputs, stream=stream)
        h_out.copy_(d_out, non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
    stream.synchronize()
    # eager: every API call issued from the host per step
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for i in range(E):
            e2e_step(i)
        b.record(stream)
    torch.cuda.synchronize(dev)
    e2e_eager_ms = a.elapsed_time(b) / E
    # the same calls captured once in a CUDA graph (copies included)
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge, stream=stream):
        for i in range(E):
            e2e_step(i)
    with torch.cuda.stream(stream):
        ge.replay()
        a.record(stream)
        ge.replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = a.elapsed_time(b) / E
    del ge
    e2e_ms, e2e_eager_ms = max_over_ranks([e2e_ms, e2e_eager_ms], world, dev)

    ms_step = ms / K
    tokens_s = tokens_per_second(world, wl.M, ms_step)
    nb = step_bytes(wl)
    path = B.pre_attn_path(dw.runner.handle, wl.M)
    gemm = path in (B.PA_PATH_GEMM_SINGLE, B.PA_PATH_GEMM_PAIR)
    kname = {B.PA_PATH_GEMV: "gemv", B.PA_PATH_GEMV_FUSED: "gemv_fused", B.PA_PATH_GEMM_SINGLE: "gemm",
             B.PA_PATH_GEMM_PAIR: "gemm2"}[path]
    kdesc = {"gemv": "pa::gemv_kernel<.., false> (tcgen05 GEMV, one cluster per head, after the prologue)",
             "gemv_fused": "pa::gemv_kernel<.., true> (prologue + tcgen05 GEMV in one kernel, one cluster per head)",
             "gemm": "pa::gemm_kernel (tcgen05, 128x128 tiles)",
             "gemm2": "pa::g2::gemm2_kernel (tcgen05 cta_group::2, 256x256 tiles)"}[kname]
    launches_per_step = 1 if path == B.PA_PATH_GEMV_FUSED else 2
    if gemm:
        achieved = step_flops(wl) / (main_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"] * FP8_OVER_BF16
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(kname, args.workload),
                "kernel": f"{kdesc}, {main_ms * 1e3:.2f} us/launch",
                "peak_source": f"{peak_src} bf16 x nominal FP8/BF16 ratio 2"}
    else:
        achieved = nb["main"] / (main_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(kname, args.workload),
                "kernel": f"{kdesc}, {main_ms * 1e3:.2f} us/launch, {nb['main']} algorithmic bytes",
                "peak_source": f"{peak_src} hbm_gbs"}
    step_roof = (nb["step"] / (ms_step * 1e-3) / 1e9) / peaks["hbm_gbs"]
    line = {
        "metric": METRIC, "value": round(tokens_s, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_step, "us_per_layer": round(ms_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 (bf16 in/out)", "data": "synthetic (seeded, configs' shapes; random-init weights)",
        "config": {"workload": args.workload, "hidden": wl.H, "nkv": wl.nkv, "M": wl.M, "N": wl.N,
                   "weight": wl.weight_fmt, "cache": wl.cache_fmt, "path": kdesc,
                   "l2": f"{copies} rotating weight+input copies ({copies * per_copy / 1e6:.0f} MB > 2x L2)",
                   "timing": "CUDA graph of K steps, PDL chained", "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "step_hbm_frac": round(step_roof, 4),
        "gpu_launches": launches_per_step * K,
        "e2e": {"value": round(tokens_per_second(world, wl.M, min(e2e_ms, e2e_eager_ms)), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E,
                "how": "pinned host inputs -> device (one copy), pre_attn_run, outputs -> pinned host (one copy), "
                       "every step; the faster of the calls issued eagerly and the same calls captured in a CUDA "
                       "graph (" + ("graph" if e2e_ms <= e2e_eager_ms else "eager") + ")",
                "graph_value": round(tokens_per_second(world, wl.M, e2e_ms), 1),
                "eager_value": round(tokens_per_second(world, wl.M, e2e_eager_ms), 1)},
        "clocks": clocks,
    }
    if gemm:
        line["step_fp8_frac"] = round(step_flops(wl) / (ms_step * 1e-3) / 1e12 / (peaks["bf16_tflops"] * FP8_OVER_BF16), 4)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, st, budget_s=args.cpu_budget)
    return line


# ------------------------------------------------------------ oracle (CPU)

def cpu_baseline(wl, st, budget_s: float = 15.0, threads: int = 1):
    """The CPU oracle as it stands, on a bounded sample of the workload's rows."""
    import oracle

    oracle.build()
    ref = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in st.items()}
    rows_done, t0 = 0, time.perf_counter()
    r = 0
    while time.perf_counter() - t0 < budget_s:
        oracle.run_rows(wl, ref, [r % wl.M], threads=threads)
        rows_done += 1
        r += 1
    dt = time.perf_counter() - t0
    return {"value": round(rows_done / dt, 3), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows_done} token rows of the {wl.name} step, one at a time, single-threaded, {dt:.1f} s"}


def run_reference(args, wl):
    import oracle

    oracle.build()
    st = workloads.host_state(wl)
    ref = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in st.items()}
    # one step = one token row of the workload (the full prologue, projection
    # and head epilogue of that token); the steps timed are capped so the run
    # stays within the budget
    t0 = time.perf_counter()
    for i in range(min(args.warmup, 3)):
        oracle.run_rows(wl, ref, [i % wl.M], threads=1)
    t_row = (time.perf_counter() - t0) / max(1, min(args.warmup, 3))
    steps = max(1, min(args.steps, int(args.cpu_budget * 4 / max(t_row, 1e-6))))
    t0 = time.perf_counter()
    for i in range(steps):
        oracle.run_rows(wl, ref, [i % wl.M], threads=1)
    dt = time.perf_counter() - t0
    v = steps / dt
    sample = f"{steps} of the {args.steps} requested steps timed; a step = one token row of {wl.name}, single-threaded"
    return {"metric": METRIC, "value": round(v, 3), "unit": "tokens/s", "n_gpus": args.gpus, "steps": steps,
            "warmup": args.warmup, "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64/f32 (CPU oracle)", "data": "synthetic",
            "config": {"workload": args.workload, "hidden": wl.H, "nkv": wl.nkv, "M": wl.M, "N": wl.N,
                       "weight": wl.weight_fmt, "cache": wl.cache_fmt},
            "impl": "reference",
            "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference", "ours"])
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--gemm", default="auto", choices=["auto", "single", "pair"],
                    help="tensor-core path tiling (auto: chosen per shape)")
    ap.add_argument("--fuse", action="store_true",
                    help="skinny path in one kernel (row normalisation inside the GEMV) where the shape allows")
    args = ap.parse_args()
    wl = get_workload(args.workload)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, wl)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from indexer_projection_gb300 import build as _b
    if rank == 0:
        _b.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    line = run_ours(args, wl, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
