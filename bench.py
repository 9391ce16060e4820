#!/usr/bin/env python
"""Benchmark of the MiniMax-M3 pre-attention step on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--workload decode|spec_decode|prefill|tiny|sweep_m<M>]
                  [--also prefill,spec_decode,index_spec_decode,drafter_spec_decode|none]

A step is one pre_attn_run() (prologue + skinny GEMV or tcgen05 GEMM with the
fused head epilogue) over one batch of the workload's synthetic inputs.  The
timed region is a CUDA graph of exactly K steps; step i uses the i-th of C
rotating copies of the layer weights and inputs (C chosen so the copies
exceed twice the L2), so weights stream from HBM as they would across layers.
Rank 0 prints one JSON line: the headline workload (decode by default) and,
under their names, the workloads of --also timed in the same run (prefill
and speculative decode: their own graphs of steps, at least a second of
them, each with its own clock record; the indexer scores of the
speculative-decode shape: a graph of pre_attn_index_scores launches; the
drafter's attention at that shape: graphs of pre_attn_drafter_attention
calls).
Under torchrun each rank runs an independent replica (the step has no
cross-GPU exchange) and the slowest rank's time sets the aggregate tokens/s.

--impl reference times the CPU oracle (tests only use it otherwise) on one
host core on bounded samples of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
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


def workload_config(name: str, wl, world: int) -> dict:
    """The workload as both arms name it (identical keys and values)."""
    return {"workload": name, "hidden": wl.H, "nkv": wl.nkv, "M": wl.M, "N": wl.N, "weight": wl.weight_fmt,
            "cache": wl.cache_fmt, "parallelism": f"replicas x{world}"}


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


# sources each kernel is compiled from (ties an ncu summary under profiles/ to them)
KERNEL_SOURCES = {"skinny": ("pa_gemv.cu", "pa_device.cuh", "pa_tc.cuh", "pa_norm.cuh"),
                  "skinny_persist": ("pa_gemv_persist.cu", "pa_device.cuh", "pa_tc.cuh", "pa_tma.h"),
                  "gemm": ("pa_gemm.cu", "pa_device.cuh", "pa_tc.cuh"),
                  "gemm_pair": ("pa_gemm2.cu", "pa_device.cuh", "pa_tc.cuh"),
                  "prologue": ("pa_prologue.cu", "pa_device.cuh", "pa_norm.cuh"),
                  "index_scores": ("pa_index.cu", "pa_device.cuh", "pa_tma.h"),
                  "drafter_attn": ("pa_drafter.cu", "pa_device.cuh", "pa_tc.cuh", "pa_tma.h")}


def kernel_sha(kernel: str) -> str:
    """Hash of the sources a kernel is built from."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "indexer_projection_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary
    profiles/<kernel>_<workload>.md, if it was taken on the current sources."""
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

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.period = period_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period), "-i", str(self.gpu)],
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
        """Clocks of the samples taken between t0 and t1 (all samples, and
        "window": "run", when the window was too short to hold one)."""
        sel = [p for (t, p) in self.samples if (t0 is None or t >= t0) and (t1 is None or t <= t1)]
        window = "timed region"
        if not sel:
            sel = [p for (_, p) in self.samples]
            window = "run"
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
                "reasons": sorted(reasons), "samples": len(sel), "window": window}


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


def path_info(B, path):
    name = {B.PA_PATH_GEMV: "skinny", B.PA_PATH_GEMV_FUSED: "skinny", B.PA_PATH_GEMV_PERSIST: "skinny_persist",
            B.PA_PATH_GEMM_SINGLE: "gemm", B.PA_PATH_GEMM_PAIR: "gemm_pair"}[path]
    desc = {B.PA_PATH_GEMV: "pa_prologue_rows_kernel then pa_skinny_proj_kernel (tcgen05 GEMV, a cluster per head), "
                            "PDL-chained",
            B.PA_PATH_GEMV_FUSED: "pa_skinny_proj_kernel with the row normalisation inside (one launch)",
            B.PA_PATH_GEMV_PERSIST: "pa_prologue_rows_kernel then pa_skinny_persist_kernel (tcgen05 GEMV, resident "
                                    "clusters walking the heads, weights double-buffered), PDL-chained",
            B.PA_PATH_GEMM_SINGLE: "pa_prologue_kernel then pa_gemm_kernel (tcgen05, 128x128 tiles)",
            B.PA_PATH_GEMM_PAIR: "pa_prologue_kernel then pa_gemm_pair_kernel (tcgen05 cta_group::2, 256x256 tiles)"}[path]
    launches = 1 if path == B.PA_PATH_GEMV_FUSED else 2
    return name, desc, launches


def build_graphs(torch, dw, n_steps, stream, events=None, lead=0):
    """CUDA graphs holding exactly n_steps timed steps (chunks of at most
    4096).  With `events` (a start / end pair, n_steps <= 4096) the one graph
    holds `lead` untimed warm-up steps, then the start event, the n_steps
    steps and the end event, so the events bracket exactly the steps' device
    execution and not the graph's launch.  The start event is recorded on a
    branch that waits for the last warm-up step: the main chain keeps its
    programmatic (PDL) edge into the first timed step, which therefore runs as
    every later one does, and the region is the span from the end of the
    last warm-up step to the end of the last timed one (n_steps step
    periods)."""
    G = min(n_steps, 4096)
    full, rest = divmod(n_steps, G)
    graphs = []
    side = torch.cuda.Stream(stream.device) if events else None
    for n in [G] * min(full, 1) + ([rest] if rest else []):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            if events:
                for i in range(lead):
                    dw.step(i, stream)
                side.wait_stream(stream)
                events[0].record(side)
            for i in range(n):
                dw.step(lead + i if events else i, stream)
            if events:
                events[1].record(stream)
                stream.wait_stream(side)
        graphs.append(g)
    order = [graphs[0]] * full + ([graphs[-1]] if rest else [])
    return graphs, order


def main_kernel_ms(torch, B, dw, stream, P):
    """Median device time of the step's main kernel with events recorded
    around it on the launching stream.  The steps are queued behind a GPU
    sleep long enough that the host never starves the GPU between them; the
    events stop the main kernel from overlapping the prologue, so this is the
    kernel alone, not its share of the pipelined step."""
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
    return statistics.median(a.elapsed_time(b) for a, b in evs[P // 4:])


def measure(args, wl, dev, world, K, W, min_seconds=0.0, flags=0):
    """Time K steps of `wl` in CUDA graphs (repeated until at least
    min_seconds when asked), the main kernel alone, and the clocks."""
    import torch
    import torch.distributed as dist

    from indexer_projection_gb300 import binding as B

    st = workloads.host_state(wl)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_copy = step_bytes(wl)["weights"] + 2 * wl.M * wl.H * 2
    copies = max(2, min(64, math.ceil(2.5 * l2 / per_copy)))
    dw = DeviceWorkload(wl, st, copies, dev, flags=flags)
    stream = torch.cuda.Stream(dev)
    path = B.pre_attn_path(dw.runner.handle, wl.M)
    sampler = ClockSampler(dev.index)
    sampler.start()
    with torch.cuda.stream(stream):
        for i in range(W):
            dw.step(i, stream)
    stream.synchronize()
    # one graph replayed once (K <= 4096, no minimum duration): the timing
    # events are its first and last nodes; otherwise they are recorded on
    # the stream around the replays
    inside = K <= 4096 and min_seconds <= 0
    ev_in = ((torch.cuda.Event(enable_timing=True, external=True),
              torch.cuda.Event(enable_timing=True, external=True)) if inside else None)
    graphs, order = build_graphs(torch, dw, K, stream, events=ev_in, lead=max(W, 3) if inside else 0)
    with torch.cuda.stream(stream):
        for g in graphs:  # untimed replay: instantiation / first-launch costs
            g.replay()
    stream.synchronize()
    # repeats of the K-step region, when a region alone is too short to be seen by the clock sampler
    reps = 1
    if min_seconds > 0:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for g in order:
                g.replay()
            e1.record(stream)
        stream.synchronize()
        reps = max(1, math.ceil(min_seconds * 1e3 / max(e0.elapsed_time(e1), 1e-3)))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        # the region starts behind a short GPU sleep, so the host has queued
        # the graph launches before the first event fires (device time of the
        # steps, not the host's launch latency)
        torch.cuda._sleep(int(200e-6 * 2.1e9))
        e0.record(stream)
        for _ in range(reps):
            for g in order:
                g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    region_ms = ev_in[0].elapsed_time(ev_in[1]) if inside else e0.elapsed_time(e1)
    ms = max_over_ranks([region_ms], world, dev)[0] / reps / K  # per step
    time.sleep(3 * sampler.period / 1000)
    clocks = sampler.summary(t_wall0, t_wall1)
    sampler.stop()
    del graphs, order
    main_ms = main_kernel_ms(torch, B, dw, stream, min(max(K, 50), 400))
    return dict(st=st, dw=dw, stream=stream, path=path, ms=ms, reps=reps, main_ms=main_ms, clocks=clocks,  # ms: per step
                copies=copies, per_copy=per_copy, events_inside=inside)


def end_to_end(torch, wl, st, dw, stream, E, world, dev):
    """Through the public API: pinned host inputs in, results out, every
    step.  The step's inputs sit in one pinned host block and one device
    block (ar | res | positions | slots, each 256-byte aligned), its outputs
    in one device block and one pinned host block: one copy each way per step
    (per-copy overhead, not bytes, dominated nine copies)."""
    from indexer_projection_gb300.runner import PreAttn

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
    eager_ms = a.elapsed_time(b) / E
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
    graph_ms = a.elapsed_time(b) / E
    del ge
    # pipelined, as a serving loop runs it: step i's input copy and step
    # i - 1's output copy on their own streams (a copy engine each way) while
    # step i - 1 computes; three sets of device buffers (and host output
    # buffers), events for every hand-over; every step still copies its own
    # inputs in and its results out inside the timed region.  (Two copy
    # streams each way measured the same: the copies are not latency-bound.)
    S = 3
    sets = []
    for _ in range(S):
        di = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        do = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        ho = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
        o = dict(zip(out_keys, views(do, out_offs, out_like)))
        sets.append({"di": di, "in": views(di, in_offs, src_in), "do": do, "ho": ho,
                     "out": PreAttn.outputs(o.get("residual"), o.get("q"), o.get("q_fp8"), o.get("iq"),
                                            o.get("iq_fp8"), wl.q_fp8_scale),
                     "in_done": torch.cuda.Event(), "comp_done": torch.cuda.Event(), "out_done": torch.cuda.Event()})
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def pipelined(n):
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(n):
            z = sets[i % S]
            if i >= S:
                s_in.wait_event(z["comp_done"])    # step i - S has read this input buffer
                stream.wait_event(z["out_done"])   # and its results have left this output buffer
            with torch.cuda.stream(s_in):
                z["di"].copy_(h_in, non_blocking=True)
                z["in_done"].record(s_in)
            stream.wait_event(z["in_done"])
            d_ar_i, d_res_i, d_pos_i, d_slot_i = z["in"]
            Li = dw.layers[i % len(dw.layers)]
            dw.runner.run(wl.M, d_ar_i, d_res_i, d_pos_i, d_slot_i, Li["wt"], dw.caches, z["out"], stream=stream)
            z["comp_done"].record(stream)
            s_out.wait_event(z["comp_done"])
            with torch.cuda.stream(s_out):
                z["ho"].copy_(z["do"], non_blocking=True)
                z["out_done"].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    with torch.cuda.stream(stream):
        pipelined(3 * S)
    torch.cuda.synchronize(dev)
    gp = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gp, stream=stream):
        pipelined(E)
    with torch.cuda.stream(stream):
        gp.replay()
        a.record(stream)
        gp.replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    pipe_ms = a.elapsed_time(b) / E
    del gp
    graph_ms, eager_ms, pipe_ms = max_over_ranks([graph_ms, eager_ms, pipe_ms], world, dev)
    best = min(graph_ms, eager_ms, pipe_ms)
    how = "graph" if best == graph_ms else "eager" if best == eager_ms else "pipelined graph"
    return {"value": round(tokens_per_second(world, wl.M, best), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E,
            "how": "pinned host inputs -> device (one copy), pre_attn_run, outputs -> pinned host (one copy), every "
                   "step; the fastest of: the calls issued eagerly on one stream, the same captured in a CUDA graph, "
                   "and a pipelined graph (input and output copies on their own streams, three buffer sets, so "
                   "step i's copies overlap step i - 1's kernels) (" + how + ")",
            "graph_value": round(tokens_per_second(world, wl.M, graph_ms), 1),
            "eager_value": round(tokens_per_second(world, wl.M, eager_ms), 1),
            "pipelined_value": round(tokens_per_second(world, wl.M, pipe_ms), 1)}


def roofline(B, wl, name, m, peaks, peak_src, workload_name):
    """The roofline object of the step's dominant kernel.

    Tensor-core path: the GEMM dominates the step (over 80% of it), so its
    own time (events around it) over 2MNK.  Skinny path: the step is a
    latency chain of two PDL-overlapped kernels around one HBM stream, and
    events around the GEMV stop that overlap (the kernel timed that way runs
    longer than the whole pipelined step), so the figure is the step's:
    algorithmic bytes of the step over the step time; the GEMV alone is
    reported beside it, labelled."""
    ms_step, main_ms = m["ms"] / 1.0, m["main_ms"]
    _, desc, _ = path_info(B, m["path"])
    nb = step_bytes(wl)
    if name in ("gemm", "gemm_pair"):
        achieved = step_flops(wl) / (main_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"] * FP8_OVER_BF16
        return {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(name, workload_name),
                "kernel": f"{name}: {main_ms * 1e3:.2f} us/launch (events around it), 2*M*N*K = {step_flops(wl)} FLOP",
                "peak_source": f"{peak_src} bf16 x nominal FP8/BF16 ratio 2 (of measured)"}
    achieved = nb["step"] / (ms_step * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    # the step's DRAM bytes: the GEMV's and its row prologue's captures
    t_main, t_pro = ncu_traffic(name, workload_name), ncu_traffic("prologue", workload_name + "_rows")
    traffic = t_main + t_pro if t_main is not None and t_pro is not None else None
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "kernel": f"whole step ({desc}): {nb['step']} algorithmic bytes over {ms_step * 1e3:.3f} us",
            "main_kernel_alone": {"us": round(main_ms * 1e3, 3), "frac": round(nb["main"] / (main_ms * 1e-3) / 1e9 / peak, 4),
                                  "note": "the GEMV timed with events around it, which stops its overlap with the "
                                          "prologue; not a share of the pipelined step"},
            "peak_source": f"{peak_src} hbm_gbs (of measured)"}


def secondary(args, name, dev, world, peaks, peak_src):
    """A second workload of the same run (prefill): its own graph of steps
    (at least a second of them), main kernel and clocks."""
    import torch

    from indexer_projection_gb300 import binding as B

    wl = get_workload(name)
    K2 = 200  # a graph of this many steps, replayed for at least a second (few graph boundaries)
    m = measure(args, wl, dev, world, K2, max(3, args.warmup), min_seconds=1.0)
    kname, desc, _ = path_info(B, m["path"])
    ms = m["ms"]
    # a region of over half a second runs at the power-capped sustained
    # clock: its steps are compared with the sustained peak (the burst one
    # is reported beside it)
    region_s = ms * 1e-3 * K2 * m["reps"]
    burst = peaks["bf16_tflops"] * FP8_OVER_BF16
    sustained = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * FP8_OVER_BF16
    fp8_peak = sustained if region_s >= 0.5 else burst
    out = {"config": workload_config(name, wl, world), "path": desc, "steps": K2 * m["reps"],
           "timed_as": f"{m['reps']} replays of a CUDA graph of {K2} steps ({region_s:.2f} s)",
           "us_per_layer": round(ms * 1e3, 3), "tokens_per_s": round(tokens_per_second(world, wl.M, ms), 1),
           "step_fp8_frac": round(step_flops(wl) / (ms * 1e-3) / 1e12 / fp8_peak, 4),
           "step_fp8_peak": {"value": round(fp8_peak, 1),
                             "source": ("sustained" if region_s >= 0.5 else "burst") + " bf16 of measured x 2"},
           "step_fp8_frac_of_burst": round(step_flops(wl) / (ms * 1e-3) / 1e12 / burst, 4),
           "step_hbm_frac": round(step_bytes(wl)["step"] / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
           "roofline": roofline(B, wl, kname, m, peaks, peak_src, name), "clocks": m["clocks"]}
    del m
    torch.cuda.empty_cache()
    return out


def index_bytes(iw, st, init, local) -> int:
    """Algorithmic bytes of one indexer-score launch: each scored key block
    read once (16 KB), the index_q rows, the block table and lengths, and
    every score column written (4 bytes, -inf included)."""
    total = iw.M * 128 * 2 + st["block_table"].nbytes + st["seq_lens"].nbytes
    for r in range(iw.R):
        seq = int(st["seq_lens"][r])
        rows_p = [seq - iw.q_len + i for i in range(iw.q_len)]
        need = set()
        for p in rows_p:
            nb = p // 128 + 1
            total += nb * 128 * 4
            need |= {b for b in range(nb) if init <= b < nb - local}
        total += len(need) * 128 * 128
    return total


def index_secondary(args, name, dev, world, peaks):
    """The indexer scores of a configuration's shape, timed on their own: a
    CUDA graph of launches over keys larger than L2."""
    import torch

    from indexer_projection_gb300 import binding as B

    iw = workloads.INDEX_CONFIGS[name]()
    st = workloads.index_host_state(iw)
    init, local = iw.init_blocks, iw.local_blocks
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    d = {k: t(st[k].view(np.int16) if k == "iq" else st[k]) for k in ("iq", "index_cache", "block_table", "seq_lens")}
    cols = iw.bt_width * 128
    scores = torch.empty(iw.M, cols, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = B.pre_attn_index_scale_log2e(iw.sm_scale)
    a = B.pa_index_args(B.ptr(d["iq"]), 128 * iw.n_iq, iw.head, B.ptr(d["index_cache"]), d["index_cache"].numel() // 128,
                        B.ptr(d["block_table"]), B.ptr(d["seq_lens"]), iw.R, iw.q_len, iw.bt_width, init, local,
                        scale, B.ptr(scores), cols, B.ptr(status))
    stream = torch.cuda.Stream(dev)
    K = max(20, min(args.steps, 200))
    sampler = ClockSampler(dev.index)
    sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(5):
            B.pre_attn_index_scores(a, stream)
        g = torch.cuda.CUDAGraph()
    stream.synchronize()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(K):
            B.pre_attn_index_scores(a, stream)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 1
    t0 = time.time()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(200e-6 * 2.1e9))
        e0.record(stream)
        g.replay()
        e1.record(stream)
    stream.synchronize()
    reps = max(1, math.ceil(1.0e3 / max(e0.elapsed_time(e1), 1e-3)))
    t0 = time.time()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(200e-6 * 2.1e9))
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    t1 = time.time()
    ms = max_over_ranks([e0.elapsed_time(e1)], world, dev)[0] / (reps * K)
    time.sleep(0.06)
    clocks = sampler.summary(t0, t1)
    sampler.stop()
    nbytes = index_bytes(iw, st, init, local)
    achieved = nbytes / (ms * 1e-3) / 1e9
    del g
    return {"config": {"workload": name, "requests": iw.R, "q_len": iw.q_len, "bt_width": iw.bt_width,
                       "seq_lens": f"U[{iw.seq_lo}, {iw.seq_hi})", "init_blocks": init, "local_blocks": local},
            "kernel": "pa_index_scores_kernel (TMA key blocks, ldmatrix + mma.sync bf16)",
            "us_per_launch": round(ms * 1e3, 3), "launches": reps * K,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": ncu_traffic("index_scores", name),
                         "algorithmic_bytes": nbytes},
            "status": int(status.item()), "clocks": clocks}


def drafter_windows(dw, st):
    """Keys lo .. hi of each request's window (first row's window start,
    below seq_len, at most max_blocks blocks from lo's block)."""
    out = []
    for r in range(dw.R):
        p0 = int(st["positions"][r * dw.q_len])
        lo = max(p0 - (dw.window - 1), 0)
        hi = min(int(st["seq_lens"][r]) - 1, (lo // 128 + dw.max_blocks) * 128 - 1)
        out.append((lo, hi))
    return out


def drafter_accounting(dw, st) -> dict:
    """Algorithmic bytes and tensor FLOPs of one drafter call: the window's
    K and V bytes read once, the projection rows read, the new keys written,
    the MXFP8 output and scales written, the metadata read; QK^T and PV over
    every (row, head, window key)."""
    keys = sum(hi - lo + 1 for lo, hi in drafter_windows(dw, st) if hi >= lo)
    blocks = sum(hi // 128 - lo // 128 + 1 for lo, hi in drafter_windows(dw, st) if hi >= lo)
    M = dw.M
    attn = keys * 256 + blocks * 4 + dw.R * 4 + M * 8 + M * 2048 + M * 64
    qkv = M * 18 * 128 * 2 + M * 256 + M * 16 + M * 64 * 2 + 2 * 128 * 2
    flops = 2 * 2 * 16 * dw.q_len * keys * 128
    return {"keys": keys, "attn_bytes": attn, "call_bytes": attn + qkv, "flops": flops}


def drafter_secondary(args, name, dev, world, peaks, peak_src):
    """The drafter's attention at a configuration's shape: a CUDA graph of
    whole calls (both kernels) rotating over copies of the drafter cache and
    inputs larger than twice the L2, and a graph of the attention kernel
    alone (its q8 rows and new keys already in place) for its roofline."""
    import torch

    from indexer_projection_gb300 import binding as B

    dw = workloads.DRAFTER_CONFIGS[name]()
    st = workloads.drafter_host_state(dw)
    acc = drafter_accounting(dw, st)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_copy = st["cache"].nbytes + st["qkv"].nbytes
    copies = max(2, math.ceil(2 * l2 / per_copy) + 1)
    shared = {k: t(st[k]) for k in ("positions", "slot_mapping", "block_table", "seq_lens")}
    shared["qn"], shared["kn"] = t(st["qn"].view(np.int16)), t(st["kn"].view(np.int16))
    shared["cos_sin"] = t(st["cos_sin"].view(np.int16))
    M = dw.M
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pb = B.pre_attn_drafter_part_blocks(dw.R, dw.max_blocks, sms)
    wsb = B.pre_attn_drafter_workspace_bytes(dw.R, dw.max_blocks, pb)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    codes = torch.empty(M, 2048, dtype=torch.uint8, device=dev)
    scales = torch.empty(M, 64, dtype=torch.uint8, device=dev)
    bufs, args_full, args_attn = [], [], []
    for c in range(copies):
        cache, qkv = t(st["cache"]), t(st["qkv"].view(np.int16))
        q8 = torch.empty(M * 16, 128, dtype=torch.uint8, device=dev)
        bufs.append((cache, qkv, q8))
        for with_qkv, lst in ((True, args_full), (False, args_attn)):
            a = B.pa_drafter_args()
            if with_qkv:
                a.qkv, a.qkv_stride = B.ptr(qkv), qkv.shape[1]
                a.qn, a.kn, a.eps = B.ptr(shared["qn"]), B.ptr(shared["kn"]), dw.eps
                a.cos_sin, a.max_pos = B.ptr(shared["cos_sin"]), shared["cos_sin"].shape[0]
                a.slot_mapping = B.ptr(shared["slot_mapping"])
            a.positions = B.ptr(shared["positions"])
            a.cache, a.num_blocks = B.ptr(cache), cache.shape[0]
            a.block_table, a.bt_width = B.ptr(shared["block_table"]), shared["block_table"].shape[1]
            a.seq_lens, a.R, a.q_len = B.ptr(shared["seq_lens"]), dw.R, dw.q_len
            a.window, a.max_blocks, a.part_blocks, a.sm_scale = dw.window, dw.max_blocks, pb, dw.sm_scale
            a.q8, a.out_codes, a.out_scales = B.ptr(q8), B.ptr(codes), B.ptr(scales)
            a.workspace, a.workspace_bytes, a.status = B.ptr(ws), wsb, B.ptr(status)
            lst.append(a)
    stream = torch.cuda.Stream(dev)
    K = max(20, min(args.steps, 200))
    sampler = ClockSampler(dev.index)
    sampler.start()

    def timed(arg_list):
        with torch.cuda.stream(stream):
            for i in range(5):
                B.pre_attn_drafter_attention(arg_list[i % copies], stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(K):
                B.pre_attn_drafter_attention(arg_list[i % copies], stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
        reps = max(1, math.ceil(0.5e3 / max(e0.elapsed_time(e1), 1e-3)))
        t0 = time.time()
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(200e-6 * 2.1e9))
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        stream.synchronize()
        t1 = time.time()
        ms = max_over_ranks([e0.elapsed_time(e1)], world, dev)[0] / (reps * K)
        del g
        return ms, reps * K, t0, t1

    # the full calls first: they write every copy's q8 rows and new keys,
    # which the attention-only graph then reads
    ms_call, n_call, t0, _ = timed(args_full)
    ms_att3, n_attn, _, t1 = timed(args_attn)
    # the attention kernel alone: events recorded around it, calls queued
    # behind a GPU sleep so the host never starves the GPU between them
    P = 64
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(P)]
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            e0.record(stream)
            e1.record(stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(2e-3 * 2.1e9))
        for i, (e0, e1) in enumerate(evs):
            a = args_attn[i % copies]
            a.prof_before, a.prof_after = e0.cuda_event, e1.cuda_event
            B.pre_attn_drafter_attention(a, stream)
            a.prof_before, a.prof_after = None, None
    stream.synchronize()
    ms_attn = max_over_ranks([statistics.median(e0.elapsed_time(e1) for e0, e1 in evs[P // 4:])], world, dev)[0]
    time.sleep(0.06)
    clocks = sampler.summary(t0, t1)
    sampler.stop()
    hbm = peaks["hbm_gbs"]
    fp8 = peaks["bf16_tflops"] * FP8_OVER_BF16
    a_gbs = acc["attn_bytes"] / (ms_attn * 1e-3) / 1e9
    c_gbs = acc["call_bytes"] / (ms_call * 1e-3) / 1e9
    out = {"config": {"workload": name, "requests": dw.R, "q_len": dw.q_len, "window": dw.window,
                      "max_blocks": dw.max_blocks, "part_blocks": pb, "seq_lens": f"U[{dw.seq_lo}, {dw.seq_hi})",
                      "window_keys": acc["keys"]},
           "kernels": "pa_drafter_qkv_kernel (head norm, RoPE, FP8, cache insert) + pa_drafter_attn_kernel "
                      "(tcgen05 S = QK^T, O += PV in TMEM, TMA K/V from the cache) + pa_drafter_merge_kernel "
                      "(ordered merge, bf16, MXFP8)",
           "l2": f"{copies} rotating cache + input copies ({copies * per_copy / 1e6:.0f} MB > 2x L2)",
           "us_per_call": round(ms_call * 1e3, 3), "calls": n_call,
           "rows_per_s": round(M / (ms_call * 1e-3), 1),
           "call_hbm_frac": round(c_gbs / hbm, 4),
           "us_attention_and_merge": round(ms_att3 * 1e3, 3),
           "us_attention_kernel": round(ms_attn * 1e3, 3), "attention_timing": "median of 48 launches, "
                                  "CUDA events around the kernel on its stream",
           "roofline": {"bound": "hbm", "achieved": round(a_gbs, 1), "peak": hbm, "unit": "GB/s",
                        "frac": round(a_gbs / hbm, 4), "traffic": ncu_traffic("drafter_attn", name),
                        "algorithmic_bytes": acc["attn_bytes"], "peak_source": f"{peak_src} copy"},
           "tensor": {"achieved_tflops": round(acc["flops"] / (ms_attn * 1e-3) / 1e12, 1),
                      "peak_tflops": round(fp8, 1),
                      "frac": round(acc["flops"] / (ms_attn * 1e-3) / 1e12 / fp8, 4),
                      "peak_source": f"burst bf16 of {peak_src} x {FP8_OVER_BF16:g}"},
           "gpu_launches": 3 * n_call + 2 * n_attn + 2 * P,
           "status": int(status.item()), "clocks": clocks}
    del bufs, args_full, args_attn
    torch.cuda.empty_cache()
    return out


def run_ours(args, wl, rank, world, local_rank):
    import torch

    from indexer_projection_gb300 import binding as B

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks, peak_src = measured_peaks()
    flags = {"auto": 0, "single": B.PA_FLAG_GEMM_SINGLE, "pair": B.PA_FLAG_GEMM_PAIR}[args.gemm]
    if args.fuse:
        flags |= B.PA_FLAG_FUSE
    flags |= {"auto": 0, "regular": B.PA_FLAG_GEMV_REGULAR, "persist": B.PA_FLAG_GEMV_PERSIST}[args.gemv]
    K, W = args.steps, args.warmup
    m = measure(args, wl, dev, world, K, W, flags=flags)
    kname, desc, launches = path_info(B, m["path"])
    e2e = end_to_end(torch, wl, m["st"], m["dw"], m["stream"], min(max(K, 200), 2000), world, dev)
    ms_step = m["ms"]
    nb = step_bytes(wl)
    line = {
        "metric": METRIC, "value": round(tokens_per_second(world, wl.M, ms_step), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": ms_step, "us_per_layer": round(ms_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 (bf16 in/out)", "data": "synthetic (seeded, configs' shapes; random-init weights)",
        "config": workload_config(args.workload, wl, world),
        "path": desc,
        "l2": f"inputs larger than L2: {m['copies']} rotating weight+input copies "
              f"({m['copies'] * m['per_copy'] / 1e6:.0f} MB > 2x L2), no flush",
        "timing": ("one CUDA graph replayed once between synchronizes: max(W, 3) untimed warm-up steps, "
                   "then exactly K timed steps (PDL chained) between two CUDA event nodes; the start event "
                   "waits, on a side branch, for the last warm-up step, so the region is K step periods "
                   "from the end of that step to the end of the last timed one" if m["events_inside"] else
                   "CUDA events around CUDA graphs of exactly K steps in all (PDL chained)"),
        "roofline": roofline(B, wl, kname, m, peaks, peak_src, args.workload),
        "step_hbm_frac": round(nb["step"] / (ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
        "gpu_launches": launches * K,
        "e2e": e2e,
        "clocks": m["clocks"],
    }
    if kname in ("gemm", "gemm_pair"):
        line["step_fp8_frac"] = round(step_flops(wl) / (ms_step * 1e-3) / 1e12 /
                                      (peaks["bf16_tflops"] * FP8_OVER_BF16), 4)
    st = m["st"]
    del m
    torch.cuda.empty_cache()
    for name in [x for x in args.also.split(",") if x and x != "none" and x != args.workload]:
        if name in workloads.INDEX_CONFIGS:
            line[name] = index_secondary(args, name, dev, world, peaks)
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                line[name]["cpu_oracle"] = cpu_oracle_requests("index", name)
        elif name in workloads.DRAFTER_CONFIGS:
            line[name] = drafter_secondary(args, name, dev, world, peaks, peak_src)
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                line[name]["cpu_oracle"] = cpu_oracle_requests("drafter", name)
        else:
            line[name] = secondary(args, name, dev, world, peaks, peak_src)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, st, budget_s=args.cpu_budget)
    return line


# ------------------------------------------------------------ oracle (CPU)

def cpu_info() -> dict:
    model = platform.processor() or platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model, "machine": platform.machine()}


class OneCore:
    """Pin this process to one host core for the duration (restored after)."""

    def __enter__(self):
        self.old = None
        self.core = None
        if hasattr(os, "sched_getaffinity"):
            self.old = os.sched_getaffinity(0)
            self.core = max(self.old)  # the last core: away from core 0's interrupts
            os.sched_setaffinity(0, {self.core})
        return self

    def __exit__(self, *exc):
        if self.old is not None:
            os.sched_setaffinity(0, self.old)


def cpu_baseline(wl, st, budget_s: float = 15.0):
    """The CPU oracle as it stands, single-threaded on one pinned core, on a
    bounded sample of the workload's rows."""
    import oracle

    oracle.build()
    ref = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in st.items()}
    rows_done = 0
    with OneCore() as pin:
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            oracle.run_rows(wl, ref, [rows_done % wl.M], threads=1)
            rows_done += 1
        dt = time.perf_counter() - t0
    return {"value": round(rows_done / dt, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{rows_done} token rows of the {wl.name} step, one at a time, single-threaded on core "
                      f"{pin.core}, {dt:.1f} s", **cpu_info()}


def cpu_oracle_requests(kind, name, budget_s: float = 4.0):
    """The CPU oracle of a secondary workload (the indexer scores or the
    drafter's attention), single-threaded on one pinned core, on whole
    requests in order until the budget runs out; scaled to one call of all
    its requests by their share of the call's work (window keys or scored
    blocks)."""
    import oracle

    oracle.build()
    if kind == "index":
        iw = workloads.INDEX_CONFIGS[name]()
        st = workloads.index_host_state(iw)
        scale = float(np.float32(oracle.index_scale_log2e(iw.sm_scale)))
        work = [max(1, (int(s) - 1) // 128 + 1) for s in st["seq_lens"]]

        def one(r):
            oracle.index_scores(st["iq"][:, iw.head * 128:(iw.head + 1) * 128], st["index_cache"],
                                st["block_table"], st["seq_lens"], iw.q_len, iw.init_blocks, iw.local_blocks, scale,
                                st["block_table"].shape[1] * 128, rows=[r * iw.q_len], threads=1)
        R, unit = iw.R, "blocks"
    else:
        dw = workloads.DRAFTER_CONFIGS[name]()
        st = workloads.drafter_host_state(dw)
        cache = st["cache"].copy()
        q8 = oracle.drafter_qkv(st["qkv"], st["qn"], st["kn"], dw.eps, st["cos_sin"], st["positions"],
                                st["slot_mapping"], cache)
        work = [hi - lo + 1 for lo, hi in drafter_windows(dw, st)]
        part = 9

        def one(r):
            oracle.drafter_attention(q8, cache, st["block_table"], st["seq_lens"], st["positions"], dw.q_len,
                                     dw.window, dw.max_blocks, part, dw.sm_scale, rows=[r * dw.q_len], threads=1)
        R, unit = dw.R, "window keys"
    done, share = 0, 0
    with OneCore() as pin:
        t0 = time.perf_counter()
        while done < R and (done == 0 or time.perf_counter() - t0 < budget_s):
            one(done)
            share += work[done]
            done += 1
        dt = time.perf_counter() - t0
    us_per_call = dt * 1e6 * sum(work) / share
    return {"us_per_call": round(us_per_call, 1), "cores": 1, "kind": "oracle",
            "sample": f"{done} of {R} requests ({share} of {sum(work)} {unit}), single-threaded on core {pin.core}, "
                      f"{dt:.1f} s, scaled by {unit}"}


def run_reference(args, wl):
    import oracle

    oracle.build()
    st = workloads.host_state(wl)
    ref = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in st.items()}
    # one step = one token row of the workload (the full prologue, projection
    # and head epilogue of that token); the steps timed are capped so the run
    # stays within the budget
    with OneCore() as pin:
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
    sample = (f"{steps} of the {args.steps} requested steps timed; a step = one token row of {wl.name}, "
              f"single-threaded on core {pin.core}")
    return {"metric": METRIC, "value": round(v, 3), "unit": "tokens/s", "n_gpus": args.gpus, "steps": steps,
            "warmup": args.warmup, "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64/f32 (CPU oracle)", "data": "synthetic",
            "config": workload_config(args.workload, wl, args.gpus),
            "path": "the CPU oracle (plain C, single-threaded), one token row a step", "impl": "reference",
            "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample,
                             **cpu_info()},
            "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference", "ours"])
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--also", default="prefill,spec_decode,sweep_m8,index_spec_decode,drafter_spec_decode",
                    help="comma-separated workloads also timed in the same run, each reported under its name "
                         "(the step's configurations, or an indexer-score configuration); none: skip")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--gemm", default="auto", choices=["auto", "single", "pair"],
                    help="tensor-core path tiling (auto: chosen per shape)")
    ap.add_argument("--gemv", default="auto", choices=["auto", "regular", "persist"],
                    help="skinny GEMV grid (auto: persistent when more heads than clusters fit at once)")
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
