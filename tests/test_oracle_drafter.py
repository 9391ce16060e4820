"""Pins of the drafter-attention oracle ("vllm.models.minimax_m3.amd.mono.
drafter.attention": window, block_math / block_acc, merge_task, qkv_rows)
against what the page and the mathematics fix, without the GPU:

  - the key window, values worked out by hand from the window formula;
  - identical keys: every valid P is exactly 256, so each output row is the
    plain mean of the V rows its window admits (non-causal inside the
    request, kp > p0 + j - window per row), in any partition layout;
  - a row with one valid key returns that key's V;
  - two valid keys in one partition: (256 v_max + E4M3(p) v_other) /
    (256 + p) with p = 2^((s_other - s_max) C + 8) (P x 256, l summing the
    unquantised p), and the variant where the larger key comes second (the
    first block's o and l rescaled by alpha, unquantised);
  - two keys in two partitions: the merge is the exact softmax (no P
    quantisation at all);
  - the MXFP8 codes and scales are torch's E4M3 cast of bf16(out) / 2^e with
    the smallest e that keeps the block within 448;
  - an empty window gives zero rows; max_blocks clips the window;
  - qkv_rows: V is stored as its E4M3 cast, q with zero gamma at position 0
    is the E4M3 cast of y / rms(y), rows with slot < 0 store nothing.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads

C_SCALE = 128 ** -0.5
C = C_SCALE / math.log(2.0)


def e4m3(x):
    """torch's OCP E4M3 cast (round to nearest even), codes as uint8."""
    return torch.tensor(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def dec(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def bf16_dec(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_round(x):
    return torch.tensor(np.asarray(x, np.float64)).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def single_request(seq, q_len, nblocks, rng):
    """One request with seq keys: blocks 0 .. nblocks - 1 physical in a
    shuffled order, positions seq - q_len .. seq - 1."""
    perm = rng.permutation(nblocks).astype(np.int32)
    bt = perm[None, :].copy()
    pos = np.arange(seq - q_len, seq, dtype=np.int64)
    return bt, np.array([seq], np.int32), pos


def run(q8, cache, bt, seq, pos, q_len, window=4096, max_blocks=34, part_blocks=34):
    return oracle.drafter_attention(q8, cache, bt, seq, pos, q_len, window, max_blocks, part_blocks, C_SCALE)


@pytest.mark.parametrize("p0,seq,window,maxb,lo,hi", [
    (5000, 5007, 4096, 34, 905, 5006),    # lo = 5000 - 4095; hi = seq - 1 (block 7 + 34 blocks reach 5247)
    (10, 17, 4096, 34, 0, 16),            # the window starts before key 0
    (5000, 5007, 4096, 2, 905, 1151),     # max_blocks = 2: blocks 7 and 8 -> (7 + 2) * 128 - 1
    (5000, 100, 4096, 34, 905, 99),       # seq below lo: empty
    (300, 301, 1, 34, 300, 300),          # window 1: the first row's own key
    (127, 4230, 4096, 34, 0, 4229),       # keys 0 .. 4229 need blocks 0 .. 33
    (4223, 8230, 4096, 34, 128, 4479),    # lo = 128 (block 1): hi = (1 + 34) * 128 - 1
])
def test_window_by_hand(p0, seq, window, maxb, lo, hi):
    assert oracle.drafter_window(p0, seq, window, maxb) == (lo, hi)


def uniform_keys_case(seq, q_len, window, nblocks, rng):
    cache = e4m3(rng.standard_normal((nblocks, 128, 256)))
    kcode = e4m3(rng.standard_normal(128))
    cache[:, :, :128] = kcode  # every key the same
    bt, sl, pos = single_request(seq, q_len, nblocks, rng)
    q8 = e4m3(rng.standard_normal((q_len * 16, 128)))
    return q8, cache, bt, sl, pos


@pytest.mark.parametrize("seq,q_len,window,part", [
    (5000, 7, 4096, 34), (5000, 7, 4096, 1), (5000, 7, 4096, 5), (300, 7, 4096, 3), (4300, 8, 300, 2),
    (1000, 1, 64, 1), (5190, 7, 4096, 7),
])
def test_identical_keys_give_the_window_mean(seq, q_len, window, part):
    rng = np.random.default_rng(seq + q_len + window + part)
    nblocks = (seq + 127) // 128
    q8, cache, bt, sl, pos = uniform_keys_case(seq, q_len, window, nblocks, rng)
    out, codes, scales = run(q8, cache, bt, sl, pos, q_len, window=window, part_blocks=part)
    p0 = seq - q_len
    v = dec(cache[:, :, 128:])
    for j in range(q_len):
        first = max(p0 - window + 1, 0, p0 + j - window + 1)
        keys = np.arange(first, seq)  # every key up to seq - 1: non-causal inside the request
        rows = v[bt[0, keys // 128], keys % 128]
        want = bf16_round(rows.mean(axis=0).astype(np.float32))
        got = bf16_dec(out[j]).reshape(16, 128)
        assert np.array_equal(got, np.broadcast_to(want, (16, 128))), f"row {j}"


def test_one_valid_key_returns_its_value():
    rng = np.random.default_rng(7)
    seq, q_len = 900, 7
    nblocks = 8
    cache = e4m3(rng.standard_normal((nblocks, 128, 256)))
    bt, sl, pos = single_request(seq, q_len, nblocks, rng)
    q8 = e4m3(rng.standard_normal((q_len * 16, 128)))
    out, _, _ = run(q8, cache, bt, sl, pos, q_len, window=1)
    last = seq - 1
    want = dec(cache[bt[0, last // 128], last % 128, 128:])
    assert np.array_equal(bf16_dec(out[q_len - 1]).reshape(16, 128), np.broadcast_to(want, (16, 128)))


def two_key_case(seq, a, b, part, rng):
    """Window 2: the last row sees keys seq - 2 (score a) and seq - 1 (score b);
    q = e_0 so the score is the key's dim-0 value; V of the larger-score key
    is 0 when it is the first, so its partner's weight shows alone."""
    q_len = 3
    nblocks = (seq + 127) // 128
    cache = np.zeros((nblocks, 128, 256), np.uint8)
    bt, sl, pos = single_request(seq, q_len, nblocks, rng)
    q8 = np.zeros((q_len * 16, 128), np.uint8)
    q8[:, 0] = e4m3(1.0)
    ka, kb = seq - 2, seq - 1
    cache[bt[0, ka // 128], ka % 128, 0] = e4m3(a)
    cache[bt[0, kb // 128], kb % 128, 0] = e4m3(b)
    va = e4m3(rng.standard_normal(128))
    vb = e4m3(rng.standard_normal(128))
    cache[bt[0, ka // 128], ka % 128, 128:] = va
    cache[bt[0, kb // 128], kb % 128, 128:] = vb
    out, _, _ = run(q8, cache, bt, sl, pos, q_len, window=2, part_blocks=part)
    return bf16_dec(out[q_len - 1]).reshape(16, 128)[0], dec(va), dec(vb)


def test_two_keys_one_partition_larger_first():
    # keys in one block; s_a = 64 > s_b = -1.75: p_b = 256 * 2^(-65.75 C) ~ 0.766 -> E4M3 0.75
    rng = np.random.default_rng(11)
    got, va, vb = two_key_case(1000, 64.0, -1.75, 34, rng)
    p = np.float32(2.0 ** ((-1.75 - 64.0) * C + 8.0))
    pq = dec(e4m3(p))
    assert pq == 0.75
    want = bf16_round(((256.0 * va + pq * vb) / (256.0 + np.float64(p))).astype(np.float32))
    assert np.array_equal(got, want)


def test_two_keys_one_partition_larger_second():
    # keys 1022 and 1023 of block 7... seq = 1024: the smaller key comes first,
    # block by block in one partition: the second block raises m, alpha
    # rescales the first block's unquantised 256 and its o
    rng = np.random.default_rng(12)
    seq = 1025  # keys 1023 (block 7) and 1024 (block 8)
    got, va, vb = two_key_case(seq, -1.75, 64.0, 34, rng)
    alpha = 2.0 ** ((-1.75 - 64.0) * C)
    want = bf16_round(((alpha * 256.0 * va + 256.0 * vb) / (alpha * 256.0 + 256.0)).astype(np.float32))
    assert np.array_equal(got, want)


def test_two_keys_two_partitions_merge_exactly():
    # one key a partition: each partition's P is exactly 256, so the merge is
    # the exact softmax of the two scores
    rng = np.random.default_rng(13)
    got, va, vb = two_key_case(1025, 64.0, 60.0, 1, rng)
    w = np.array([1.0, 2.0 ** ((60.0 - 64.0) * C)])
    want = bf16_round(((w[0] * va + w[1] * vb) / w.sum()).astype(np.float32))
    assert np.array_equal(got, want)
    # the same keys in one partition quantise the second P: a different result
    got1, _, _ = two_key_case(1025, 64.0, 60.0, 34, np.random.default_rng(13))
    assert not np.array_equal(got, got1)


def test_mxfp8_codes_follow_the_bf16_output():
    rng = np.random.default_rng(21)
    seq, q_len, nblocks = 3000, 7, 24
    cache = e4m3(rng.standard_normal((nblocks, 128, 256)) * np.exp(rng.standard_normal((nblocks, 128, 1))))
    bt, sl, pos = single_request(seq, q_len, nblocks, rng)
    q8 = e4m3(rng.standard_normal((q_len * 16, 128)))
    out, codes, scales = run(q8, cache, bt, sl, pos, q_len, part_blocks=4)
    x = bf16_dec(out).reshape(q_len, 64, 32)
    amax = np.abs(x).max(axis=2)
    e = scales.astype(np.int64) - 127
    assert np.all(448.0 * np.ldexp(1.0, e) >= amax)
    assert np.all((448.0 * np.ldexp(1.0, e - 1) < amax) | (amax == 0))
    want = e4m3((x * np.ldexp(1.0, -e)[:, :, None]).astype(np.float32)).reshape(q_len, 2048)
    assert np.array_equal(codes, want)


def test_empty_window_gives_zero_rows():
    rng = np.random.default_rng(5)
    nblocks = 4
    cache = e4m3(rng.standard_normal((nblocks, 128, 256)))
    bt = np.arange(nblocks, dtype=np.int32)[None]
    pos = np.arange(5000, 5007, dtype=np.int64)  # seq far below the window start
    out, codes, scales = run(e4m3(rng.standard_normal((7 * 16, 128))), cache, bt, np.array([100], np.int32), pos, 7)
    assert not out.any() and not codes.any() and np.all(scales == 127)


def test_max_blocks_clips_the_window():
    # clipping to 2 blocks = the same keys as a cache whose later keys are gone
    rng = np.random.default_rng(6)
    seq, q_len, nblocks = 2000, 7, 16
    cache = e4m3(rng.standard_normal((nblocks, 128, 256)))
    bt, sl, pos = single_request(seq, q_len, nblocks, rng)
    q8 = np.tile(e4m3(rng.standard_normal((16, 128))), (q_len, 1))  # every row the same q
    out, _, _ = run(q8, cache, bt, sl, pos, q_len, window=4096, max_blocks=2)
    # with max_blocks = 2 from block 0 the keys are 0 .. 255 for every row
    # (the window reaches back past key 0), so all rows agree
    assert all(np.array_equal(out[0], out[j]) for j in range(q_len))
    out2, _, _ = run(q8[:16], cache, bt, np.array([256], np.int32), pos[:1] * 0 + 255, 1, window=4096)
    assert np.array_equal(out[0], out2[0])


def test_partition_layouts_agree_within_fp8_rounding():
    dw = workloads.DrafterWorkload("t", R=3, q_len=7, seq_lo=300, seq_hi=6000, seed=4, stale="nan")
    st = workloads.drafter_host_state(dw)
    cache = st["cache"].copy()
    q8 = oracle.drafter_qkv(st["qkv"], st["qn"], st["kn"], dw.eps, st["cos_sin"], st["positions"],
                            st["slot_mapping"], cache)
    outs = [run(q8, cache, st["block_table"], st["seq_lens"], st["positions"], 7, part_blocks=pb)[0]
            for pb in (1, 4, 34)]
    a = [bf16_dec(o) for o in outs]
    assert np.all(np.isfinite(a[0]))
    for b in a[1:]:
        assert np.allclose(a[0], b, rtol=5e-2, atol=2e-2)


def test_qkv_rows_store_v_and_normalise_q():
    rng = np.random.default_rng(8)
    M = 3
    qkv = workloads._bf16_bits(torch.from_numpy(rng.standard_normal((M, 18 * 128))))
    zero = np.zeros(128, np.uint16)
    cs = workloads.cos_sin_table(16)
    cache = np.full((2, 128, 256), 0xA5, np.uint8)
    slots = np.array([5, -1, 200], np.int64)
    pos = np.zeros(M, np.int64)
    q8 = oracle.drafter_qkv(qkv, zero, zero, 1e-6, cs, pos, slots, cache)
    y = bf16_dec(qkv).reshape(M, 18, 128)
    for m in range(M):
        for h in range(16):
            z = y[m, h] / np.sqrt(np.mean(y[m, h] ** 2) + 1e-6)
            assert np.array_equal(q8[m * 16 + h], e4m3(z.astype(np.float32)))
    flat = cache.reshape(-1, 256)
    assert np.array_equal(flat[5, 128:], e4m3(y[0, 17].astype(np.float32)))
    assert np.array_equal(flat[200, 128:], e4m3(y[2, 17].astype(np.float32)))
    k = y[2, 16] / np.sqrt(np.mean(y[2, 16] ** 2) + 1e-6)
    assert np.array_equal(flat[200, :128], e4m3(k.astype(np.float32)))
    untouched = np.ones(256, bool)
    untouched[[5, 200]] = False
    assert np.all(flat[untouched] == 0xA5)


def test_qkv_rows_take_their_own_gamma_and_position():
    # q heads use qn, k uses kn, v neither; RoPE reads the row's own position
    # (the head norm and RoPE themselves are pinned with the step's oracle)
    rng = np.random.default_rng(9)
    M = 3
    qkv = workloads._bf16_bits(torch.from_numpy(rng.standard_normal((M, 18 * 128))))
    qn = workloads._bf16_bits(torch.from_numpy(rng.standard_normal(128) * 0.3))
    kn = workloads._bf16_bits(torch.from_numpy(rng.standard_normal(128) * 0.3))
    cs = workloads.cos_sin_table(64)
    pos = np.array([3, 40, 17], np.int64)
    slots = np.array([0, 1, 2], np.int64)
    cache = np.zeros((1, 128, 256), np.uint8)
    q8 = oracle.drafter_qkv(qkv, qn, kn, 1e-6, cs, pos, slots, cache)
    y = bf16_dec(qkv).reshape(M, 18, 128).astype(np.float32)
    for m in range(M):
        for h in (0, 9, 15, 16):
            z = oracle.rope_neox(oracle.head_rmsnorm(y[m, h], qn if h < 16 else kn, 1e-6), cs[pos[m]])
            want = e4m3(np.asarray(z, np.float64).astype(np.float32))
            got = q8[m * 16 + h] if h < 16 else cache[0, m, :128]
            assert np.array_equal(got, want), (m, h)
        assert np.array_equal(cache[0, m, 128:], e4m3(y[m, 17]))
