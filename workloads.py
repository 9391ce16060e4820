"""Seeded synthetic workloads for the MiniMax-M3 pre-attention step.

This module only draws inputs: random bf16 activations and gammas, an FP8
weight with its scales, the RoPE cos / sin table, positions and cache slots,
and sentinel-filled caches and output buffers.  It holds none of the step's
own arithmetic; both the CUDA path and the CPU oracle consume what it makes.

Weight preparation (the weight is an input of the step, quantised offline by
the model loader) uses torch's own float8 cast on values already scaled into
[-448, 448].  The per-channel scale is amax / 448 of each output channel; the
MXFP8 block exponent is the smallest power of two that keeps the block's
amax within 448 (the same reading the step uses for its activations).
"""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128
SENTINEL = 0xA5


@dataclass
class Workload:
    name: str
    H: int
    nkv: int
    M: int
    weight_fmt: str  # "ptpc" | "mx"
    cache_fmt: str   # "fp8" | "nvfp4"
    seed: int
    n_q: int = 0     # 0 -> 16 * nkv
    n_iq: int = 0    # 0 -> nkv
    block_size: int = 16
    kv_page_stride: int = 8
    static_kv_scale: bool = False
    eps: float = 1e-6
    q_bf16: bool = True
    q_fp8: bool = False
    iq_bf16: bool = True
    iq_fp8: bool = False
    q_fp8_scale: float = 1.0
    k_global: float = 1.0
    v_global: float = 1.0
    # position / slot recipe
    positions: str = "uniform"   # uniform | spec | prefill | runs
    max_pos: int = 256
    requests: int = 0
    q_len: int = 1
    seq_len_range: tuple = (1024, 32768)
    pool_pages16: int = 64       # FP8 caches: page-16 pages (per KV head)
    pool_pages: int = 0          # NVFP4 caches: pages of block_size tokens
    page_pad: int = 0            # NVFP4: extra bytes per page (any page stride)
    outlier_frac: float = 0.0
    outlier_scale: float = 50.0
    skip_rows: tuple = ()        # rows whose slots are -1
    separate_index_slots: bool = False

    def __post_init__(self):
        if self.n_q == 0:
            self.n_q = 16 * self.nkv
        if self.n_iq == 0:
            self.n_iq = self.nkv

    @property
    def n_heads(self) -> int:
        return self.n_q + 2 * self.nkv + self.n_iq + 1

    @property
    def N(self) -> int:
        return self.n_heads * HEAD_DIM

    # FP8 cache geometry
    @property
    def num_pages16(self) -> int:
        return self.pool_pages16

    @property
    def num_index_slots(self) -> int:
        return self.pool_pages16 * 16

    # NVFP4 cache geometry
    @property
    def kv_pages(self) -> int:
        return self.pool_pages

    @property
    def kv_page_bytes(self) -> int:
        return 2 * self.nkv * self.block_size * 72 + self.page_pad

    @property
    def idx_pages(self) -> int:
        return self.pool_pages

    @property
    def idx_page_bytes(self) -> int:
        return self.block_size * 72 + self.page_pad

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five configurations of the pre-attention step's benchmark suite.
def tiny() -> Workload:
    return Workload("tiny", H=512, nkv=1, M=4, weight_fmt="ptpc", cache_fmt="fp8", seed=0,
                    positions="uniform", max_pos=256, pool_pages16=64)


def decode() -> Workload:
    return Workload("decode", H=6144, nkv=1, M=8, weight_fmt="ptpc", cache_fmt="fp8", seed=1,
                    positions="uniform", max_pos=32768, pool_pages16=4096)


def spec_decode() -> Workload:
    # 64 requests x 7 verify rows; page-128 blocks from a pool of 1024
    return Workload("spec_decode", H=6144, nkv=2, M=448, weight_fmt="ptpc", cache_fmt="fp8",
                    seed=2, positions="spec", requests=64, q_len=7, max_pos=32768,
                    seq_len_range=(1024, 32768), pool_pages16=1024 * 8)


def prefill() -> Workload:
    return Workload("prefill", H=6144, nkv=4, M=8192, weight_fmt="mx", cache_fmt="nvfp4", seed=3,
                    positions="prefill", requests=4, q_len=2048, max_pos=2048, pool_pages=1024,
                    q_bf16=True, q_fp8=True, iq_bf16=False, iq_fp8=True)


SWEEP_M = (1, 2, 4, 8, 16, 64, 256, 1024, 4096, 16384)


def sweep(M: int) -> Workload:
    q_len = 1 if M <= 16 else min(M, 512)
    return Workload(f"sweep_m{M}", H=6144, nkv=4, M=M, weight_fmt="mx", cache_fmt="fp8", seed=4,
                    positions="runs", requests=max(1, M // q_len), q_len=q_len,
                    max_pos=131072 + 512, pool_pages16=max(4096, 2 * (M // 16) + 4 * M // q_len + 64),
                    outlier_frac=0.01, q_bf16=True, q_fp8=True, iq_bf16=True, iq_fp8=True)


CONFIGS = {"tiny": tiny, "decode": decode, "spec_decode": spec_decode, "prefill": prefill}


# ------------------------------------------------------------------ drawing

def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _e4m3_bits(t: torch.Tensor) -> np.ndarray:
    return t.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def _mx_block_exponent(amax: torch.Tensor) -> torch.Tensor:
    """Smallest e with 448 * 2^e >= amax (0 where amax == 0), in [-127, 127]."""
    a = amax.to(torch.float64)
    e = torch.ceil(torch.log2(torch.where(a > 0, a, torch.ones_like(a)) / 448.0))
    e = torch.where(torch.ldexp(torch.full_like(a, 448.0), e - 1) >= a, e - 1, e)
    e = torch.where(torch.ldexp(torch.full_like(a, 448.0), e) < a, e + 1, e)
    e = torch.where(a > 0, e, torch.zeros_like(e))
    return e.clamp(-127, 127).to(torch.int64)


def cos_sin_table(max_pos: int, rotary_dim: int = 64, base: float = 10000.0) -> np.ndarray:
    """[max_pos, 64] bf16 = cos(p * theta_i) | sin(p * theta_i), i < 32,
    theta_i = base^(-2i / rotary_dim), computed in double."""
    half = rotary_dim // 2
    inv = base ** (-(np.arange(half, dtype=np.float64) * 2.0) / rotary_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    tab = np.concatenate([np.cos(ang), np.sin(ang)], axis=1)
    return _bf16_bits(torch.from_numpy(tab))


def _positions_and_slots(wl: Workload, g: torch.Generator):
    M = wl.M
    bs = 16 if wl.cache_fmt == "fp8" else wl.block_size
    pool = wl.pool_pages16 if wl.cache_fmt == "fp8" else wl.pool_pages
    if wl.positions == "uniform":
        pos = torch.randint(0, wl.max_pos, (M,), generator=g, dtype=torch.int64)
        slots = torch.randperm(pool * bs, generator=g)[:M].to(torch.int64)
    elif wl.positions == "spec":
        # per request a seq_len; the rows take positions seq_len - q_len .. seq_len - 1;
        # page-128 blocks of the block table (width 256) drawn distinct from the pool
        lo, hi = wl.seq_len_range
        seq = torch.randint(lo, hi, (wl.requests,), generator=g, dtype=torch.int64)
        pool128 = pool * 16 // 128
        perm = torch.randperm(pool128, generator=g)
        table = torch.full((wl.requests, 256), -1, dtype=torch.int64)
        nxt = 0
        pos_l, slot_l = [], []
        for r in range(wl.requests):
            p = torch.arange(int(seq[r]) - wl.q_len, int(seq[r]), dtype=torch.int64)
            for blk in sorted(set((p // 128).tolist())):
                table[r, blk] = perm[nxt]
                nxt += 1
            pos_l.append(p)
            slot_l.append(table[r, p // 128] * 128 + p % 128)
        pos, slots = torch.cat(pos_l), torch.cat(slot_l)
    elif wl.positions in ("prefill", "runs"):
        nreq = wl.requests
        perm = torch.randperm(pool, generator=g)
        nxt = 0
        pos_l, slot_l = [], []
        for r in range(nreq):
            if wl.positions == "prefill":
                start = 0
            else:
                start = int(torch.randint(0, wl.max_pos - wl.q_len, (1,), generator=g))
            p = torch.arange(start, start + wl.q_len, dtype=torch.int64)
            pages = {}
            for pg in sorted(set((p // bs).tolist())):
                pages[pg] = int(perm[nxt])
                nxt += 1
            pos_l.append(p)
            slot_l.append(torch.tensor([pages[int(x) // bs] * bs + int(x) % bs for x in p], dtype=torch.int64))
        pos, slots = torch.cat(pos_l)[:M], torch.cat(slot_l)[:M]
    else:
        raise ValueError(wl.positions)
    assert pos.numel() == M and slots.numel() == M
    slots = slots.clone()
    for r in wl.skip_rows:
        if r < M:
            slots[r] = -1
    islots = slots
    if wl.separate_index_slots:
        cap = wl.num_index_slots if wl.cache_fmt == "fp8" else wl.idx_pages * bs
        islots = torch.randperm(cap, generator=g)[:M].to(torch.int64)
        for r in wl.skip_rows:
            if r < M:
                islots[r] = -1
    return pos.numpy().copy(), slots.numpy().copy(), islots.numpy().copy()


def host_state(wl: Workload, with_outputs: bool = True) -> dict:
    """All inputs, sentinel-filled caches and output buffers as numpy arrays.

    bf16 tensors are uint16 bit patterns, FP8 / NVFP4 data are uint8 codes.
    """
    g = torch.Generator().manual_seed(wl.seed)
    H, N, M = wl.H, wl.N, wl.M
    st = {}
    ar = torch.randn(M, H, generator=g)
    res = torch.randn(M, H, generator=g)
    if wl.outlier_frac > 0 and M > 0:
        n_out = max(1, int(round(wl.outlier_frac * M)))
        rows = torch.randperm(M, generator=g)[:n_out]
        ar[rows] *= wl.outlier_scale
        res[rows] *= wl.outlier_scale
    st["ar"], st["res"] = _bf16_bits(ar), _bf16_bits(res)
    st["g_in"] = _bf16_bits(torch.randn(H, generator=g) * 0.1)
    for k in ("g_q", "g_k", "g_iq", "g_ik"):
        st[k] = _bf16_bits(torch.randn(HEAD_DIM, generator=g) * 0.1)
    wf = torch.randn(N, H, generator=g, dtype=torch.float32) / math.sqrt(H)
    if wl.weight_fmt == "ptpc":
        s = (wf.abs().amax(dim=1) / 448.0).to(torch.float32)
        s = torch.where(s > 0, s, torch.ones_like(s))
        st["w"] = _e4m3_bits(wf / s[:, None])
        st["w_scale"] = s.numpy().astype(np.float32)
    else:
        blocks = wf.view(N, H // 32, 32)
        e = _mx_block_exponent(blocks.abs().amax(dim=2))
        st["w"] = _e4m3_bits((blocks * torch.pow(2.0, -e.to(torch.float64)).to(torch.float32)[:, :, None]).view(N, H))
        st["wsf"] = (e + 127).to(torch.uint8).numpy().copy()
    st["cos_sin"] = cos_sin_table(wl.max_pos)
    pos, slots, islots = _positions_and_slots(wl, g)
    st["positions"], st["slot_mapping"] = pos, slots
    st["index_slot_mapping"] = islots
    if wl.cache_fmt == "fp8":
        P = wl.num_pages16 * wl.nkv
        st["k_cache"] = np.full(P * 2048, SENTINEL, np.uint8)
        st["v_cache"] = np.full(P * 2048, SENTINEL, np.uint8)
        st["k_scale"] = np.full(P * 16 * 4, SENTINEL, np.uint8).view(np.float32)
        st["v_scale"] = np.full(P * 16 * 4, SENTINEL, np.uint8).view(np.float32)
        st["index_cache"] = np.full(wl.num_index_slots * HEAD_DIM, SENTINEL, np.uint8)
    else:
        st["kv_cache"] = np.full(wl.kv_pages * wl.kv_page_bytes, SENTINEL, np.uint8)
        st["idx_cache"] = np.full(wl.idx_pages * wl.idx_page_bytes, SENTINEL, np.uint8)
    if with_outputs:
        st["residual"] = np.full((M, H), 0xA5A5, np.uint16)
        if wl.q_bf16:
            st["q_bf16"] = np.full((M, wl.n_q * HEAD_DIM), 0xA5A5, np.uint16)
        if wl.q_fp8:
            st["q_fp8"] = np.full((M, wl.n_q * HEAD_DIM), SENTINEL, np.uint8)
        if wl.iq_bf16:
            st["iq_bf16"] = np.full((M, wl.n_iq * HEAD_DIM), 0xA5A5, np.uint16)
        if wl.iq_fp8:
            st["iq_fp8"] = np.full((M, wl.n_iq * HEAD_DIM), SENTINEL, np.uint8)
    return st


CACHE_KEYS = ("k_cache", "v_cache", "k_scale", "v_scale", "index_cache", "kv_cache", "idx_cache")
OUTPUT_KEYS = ("residual", "q_bf16", "q_fp8", "iq_bf16", "iq_fp8")


# ------------------------------------------------------------ indexer scores

@dataclass
class IndexWorkload:
    """Inputs of the indexer scores: the step's index_q rows, an FP8 index
    cache holding every key of the requests, page-128 block tables and
    sequence lengths."""
    name: str
    R: int                 # requests
    q_len: int             # rows a request (speculative verify rows)
    seq_lo: int            # seq_lens ~ U[seq_lo, seq_hi)
    seq_hi: int
    bt_width: int          # block-table width (page-128 blocks)
    seed: int
    init_blocks: int = 1   # pinned first blocks
    local_blocks: int = 4  # pinned local window (blocks)
    sm_scale: float = 128 ** -0.5
    n_iq: int = 1          # index_q heads in the iq rows; the scores use head `head`
    head: int = 0

    @property
    def M(self) -> int:
        return self.R * self.q_len


def index_decode() -> IndexWorkload:
    # the decode configuration's shape: 8 requests, one row each, up to 32768 keys
    return IndexWorkload("index_decode", R=8, q_len=1, seq_lo=1, seq_hi=32769, bt_width=256, seed=1)


def index_spec_decode() -> IndexWorkload:
    # the speculative-decode configuration's shape: 64 requests x 7 rows, seq_lens U[1024, 32768)
    return IndexWorkload("index_spec_decode", R=64, q_len=7, seq_lo=1024, seq_hi=32768, bt_width=256, seed=2)


INDEX_CONFIGS = {"index_decode": index_decode, "index_spec_decode": index_spec_decode}


def index_host_state(iw: IndexWorkload) -> dict:
    """iq [M, n_iq*128] bf16 bits ~ N(0, 1) (a normed index_q has unit RMS);
    index_cache [blocks * 128, 128] E4M3 codes of N(0, 1) values (the unit-scale
    FP8 index keys); block_table [R, bt_width] int32 of distinct random blocks
    (-1 past a request's last block); seq_lens [R] int32."""
    g = torch.Generator().manual_seed(iw.seed)
    seq = torch.randint(iw.seq_lo, iw.seq_hi, (iw.R,), generator=g, dtype=torch.int64)
    seq = torch.maximum(seq, torch.full_like(seq, iw.q_len))
    nb = (seq + 127) // 128
    assert int(nb.max()) <= iw.bt_width
    pool = int(nb.sum()) + 16
    perm = torch.randperm(pool, generator=g)
    bt = torch.full((iw.R, iw.bt_width), -1, dtype=torch.int32)
    nxt = 0
    for r in range(iw.R):
        n = int(nb[r])
        bt[r, :n] = perm[nxt:nxt + n].to(torch.int32)
        nxt += n
    st = {"seq_lens": seq.to(torch.int32).numpy().copy(), "block_table": bt.numpy().copy()}
    st["iq"] = _bf16_bits(torch.randn(iw.M, iw.n_iq * HEAD_DIM, generator=g))
    keys = torch.randn(pool * 128, HEAD_DIM, generator=g)
    st["index_cache"] = _e4m3_bits(keys)
    return st


@dataclass
class DrafterWorkload:
    """Inputs of the drafter's attention: the drafter's projection rows (16 q
    heads, k, v; bf16), its q / k head-norm gammas, the RoPE table, R
    requests of q_len consecutive rows whose last row is the request's last
    key (positions seq_len - q_len .. seq_len - 1), page-128 block tables and
    a drafter KV cache of 256-byte key records (K then V, E4M3).

    Only the blocks from (seq_len - q_len - window) / 128 on are given
    physical blocks (a superset of what the key window can touch); the rest
    of a block-table row is -1.  Keys below seq_len - q_len hold E4M3 codes
    of N(0, 1) values (a normed key has unit RMS; V likewise); every other
    byte of the cache (the new rows' slots before the call, keys past
    seq_len, unused blocks) holds `stale`: "nan" fills them with E4M3 NaN
    codes (0x7f / 0xff), "random" with random bytes."""
    name: str
    R: int
    q_len: int
    seq_lo: int            # seq_lens ~ U[seq_lo, seq_hi)
    seq_hi: int
    seed: int
    window: int = 4096
    max_blocks: int = 34   # 4096 keys + 6 rows from any offset in a block
    part_blocks: int = 0   # 0: the library's choice for the device
    sm_scale: float = 128 ** -0.5
    eps: float = 1e-6
    stale: str = "nan"
    spare_blocks: int = 8
    prefilled: bool = False  # the new rows' keys already in the cache, q8 given (attention alone)

    @property
    def M(self) -> int:
        return self.R * self.q_len

    @property
    def bt_width(self) -> int:
        return (self.seq_hi + 127) // 128


def drafter_spec_decode() -> DrafterWorkload:
    # the speculative-decode configuration's shape: 64 requests x 7 rows, seq_lens U[1024, 32768)
    return DrafterWorkload("drafter_spec_decode", R=64, q_len=7, seq_lo=1024, seq_hi=32768, seed=2)


DRAFTER_CONFIGS = {"drafter_spec_decode": drafter_spec_decode}


def drafter_host_state(dw: DrafterWorkload) -> dict:
    """qkv [M, 18 * 128] bf16 bits ~ N(0, 1); qn, kn [128] bf16 bits ~ N(0, 0.1);
    cos_sin [seq_hi, 64] bf16 bits; positions, slot_mapping [M] int64;
    seq_lens [R] int32; block_table [R, bt_width] int32; cache [blocks, 128,
    256] uint8 (see DrafterWorkload); with `prefilled`, q8 [M * 16, 128]
    E4M3 codes."""
    g = torch.Generator().manual_seed(dw.seed)
    seq = torch.randint(dw.seq_lo, dw.seq_hi, (dw.R,), generator=g, dtype=torch.int64)
    seq = torch.maximum(seq, torch.full_like(seq, dw.q_len))
    nb = (seq + 127) // 128
    first = torch.clamp((seq - dw.q_len - dw.window) // 128, min=0)
    counts = nb - first
    pool = int(counts.sum()) + dw.spare_blocks
    perm = torch.randperm(pool, generator=g)
    bt = torch.full((dw.R, dw.bt_width), -1, dtype=torch.int32)
    nxt = 0
    for r in range(dw.R):
        a, b = int(first[r]), int(nb[r])
        bt[r, a:b] = perm[nxt:nxt + b - a].to(torch.int32)
        nxt += b - a
    M = dw.M
    pos = (seq.repeat_interleave(dw.q_len) - dw.q_len + torch.arange(dw.q_len).repeat(dw.R)).to(torch.int64)
    blk = bt[torch.arange(dw.R).repeat_interleave(dw.q_len), pos // 128].to(torch.int64)
    slots = blk * 128 + pos % 128
    if dw.stale == "nan":
        cache = torch.where(torch.rand(pool, 128, 256, generator=g) < 0.5, 0x7F, 0xFF).to(torch.uint8)
    else:
        cache = torch.randint(0, 256, (pool, 128, 256), generator=g, dtype=torch.uint8)
    # the keys already in the cache: below seq_len - q_len (below seq_len when prefilled)
    kv = _e4m3_bits(torch.randn(pool * 128, 256, generator=g)).reshape(pool, 128, 256)
    written = torch.zeros(pool, 128, dtype=torch.bool)
    for r in range(dw.R):
        a, b = int(first[r]), int(nb[r])
        n_old = int(seq[r]) - (0 if dw.prefilled else dw.q_len)
        for c in range(a, b):
            k = torch.arange(128) + c * 128
            written[int(bt[r, c])] = k < n_old
    cache[written] = torch.from_numpy(kv)[written]
    st = {
        "seq_lens": seq.to(torch.int32).numpy().copy(),
        "block_table": bt.numpy().copy(),
        "positions": pos.numpy().copy(),
        "slot_mapping": slots.numpy().copy(),
        "cache": cache.numpy().copy(),
        "qkv": _bf16_bits(torch.randn(M, 18 * HEAD_DIM, generator=g)),
        "qn": _bf16_bits(torch.randn(HEAD_DIM, generator=g) * 0.1),
        "kn": _bf16_bits(torch.randn(HEAD_DIM, generator=g) * 0.1),
        "cos_sin": cos_sin_table(dw.seq_hi),
    }
    if dw.prefilled:  # E4M3 codes of N(0, 1) q rows (a normed q has unit RMS)
        st["q8"] = _e4m3_bits(torch.randn(M * 16, HEAD_DIM, generator=g))
    return st
