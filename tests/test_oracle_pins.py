"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test checks the oracle against a library routine (torch / numpy casts and
matmuls), a closed form, an invariant of the mathematics, a brute-force or
alternative formulation, or a value printed on the pages (tests/golden).
A plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a swapped nibble) fails at least one of them.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def f32(x):
    return float(np.float32(x))


# ------------------------------------------------------------------ codecs

def test_e4m3_decode_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if np.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])


def test_e4m3_roundtrip_every_finite_code():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c


def test_e4m3_encode_matches_torch_rne_on_random_values():
    x = np.concatenate([rng.standard_normal(4000) * s for s in (1e-3, 0.05, 1.0, 30.0, 200.0)])
    x = np.clip(x, -448, 448).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    assert (got == ref).all()


def test_e4m3_ties_go_to_even_and_saturate():
    # the midpoint of two neighbouring magnitudes rounds to the even code
    for c in range(0, 126):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = (lo + hi) / 2
        assert np.float32(mid) == mid
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == want, (c, mid)
        assert oracle.e4m3_encode(-mid) == 0x80 | want
    for v in (448.0, 460.0, 480.0, 1e6, 3.0e38):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x38) == 1.0


def test_e2m1_codes_ties_and_saturation():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        v = oracle.e2m1_decode(c)
        assert abs(v) == mags[c & 7] and (v < 0) == (c >= 8 and c != 8)
        if c != 8:  # -0 encodes back to -0 (its sign is cleared later by the quantiser)
            assert oracle.e2m1_encode(v) == c
    assert oracle.e2m1_encode(-0.0) == 8
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for x, c in ties.items():
        assert oracle.e2m1_encode(x) == c, x
        assert oracle.e2m1_encode(-x) == (8 | c), x
    for x in (6.0, 6.5, 7.0, 100.0):
        assert oracle.e2m1_encode(x) == 7
    # nearest value off the midpoints
    for x in rng.uniform(0, 6, 2000).astype(np.float32):
        c = oracle.e2m1_encode(float(x))
        d = [abs(float(x) - m) for m in mags]
        assert d[c] == min(d)


def test_bf16_encode_matches_torch():
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        # exact ties: bf16 values plus half an ulp
                        (rng.standard_normal(2000).astype(np.float32).view(np.uint32) & 0xFFFF0000 | 0x8000).view(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_encode(float(v)) for v in x], np.uint16)
    assert (got == ref).all()
    for b in rng.integers(0, 0x7F80, 200):
        assert oracle.bf16_encode(oracle.bf16_decode(int(b))) == b


def test_e8m0_decode():
    for c in range(255):
        assert oracle.e8m0_decode(c) == 2.0 ** (c - 127)
    assert math.isnan(oracle.e8m0_decode(255))


# ------------------------------------------------------------ quant rules

def test_fp8_scale_rule():
    assert oracle.fp8_scale(0.0) == 1.0
    assert oracle.fp8_scale(448.0) == 1.0
    for a in rng.uniform(1e-3, 1e3, 100).astype(np.float32):
        assert oracle.fp8_scale(float(a)) == np.float32(a) / np.float32(448.0)


def test_mx_exponent_is_the_smallest_non_clipping_power():
    assert oracle.mx_exponent(0.0) == 0
    assert oracle.mx_exponent(448.0) == 0
    assert oracle.mx_exponent(f32(np.nextafter(np.float32(448), np.float32(1e9)))) == 1
    assert oracle.mx_exponent(224.0) == -1
    assert oracle.mx_exponent(3.0) == -7  # 448 / 128 = 3.5 >= 3 > 1.75
    for a in np.exp(rng.uniform(-40, 40, 2000)).astype(np.float32):
        e = oracle.mx_exponent(float(a))
        assert 448.0 * 2.0 ** e >= a > 448.0 * 2.0 ** (e - 1)


def test_nvfp4_group_max_maps_to_six_and_zero_group():
    for trial in range(300):
        v = (rng.standard_normal(16) * 10 ** rng.uniform(-1, 2)).astype(np.float32)
        gi = None if trial % 2 else float(np.float32(1.0) / np.float32(rng.uniform(0.5, 2)))
        nib, sf = oracle.nvfp4_group16(v, gi)
        k = int(np.argmax(np.abs(v)))
        assert nib[k] & 7 == 7, (v, nib, sf)          # |max| -> 6
        assert (nib[k] >= 8) == (v[k] < 0)
        # every element dequantises to within one E2M1 step of its value
        s = oracle.e4m3_decode(sf) / (1.0 if gi is None else gi)
        deq = np.array([oracle.e2m1_decode(n) for n in nib]) * s
        assert np.all(np.abs(deq - v) <= 2.0 * s + 1e-6)
    nib, sf = oracle.nvfp4_group16(np.zeros(16, np.float32), None)
    assert sf == 0x01 and not nib.any()              # scale floored at 2^-9
    v = np.zeros(16, np.float32)
    v[0], v[1] = 12.0, -1e-4                          # tiny negative -> +0
    nib, sf = oracle.nvfp4_group16(v, None)
    assert nib[1] == 0 and nib[0] == 7


def test_nvfp4_sign_clearing_matches_the_pages_word_trick():
    # the qkv_index_fused_epilogue page (_nvfp4_quant32) clears the sign of
    # zero-magnitude nibbles on packed words with w & (((w & m) + m) | m),
    # m = 0x77777777; the oracle clears them one nibble at a time
    m = 0x77777777
    for _ in range(2000):
        nibs = rng.integers(0, 16, 8)
        w = 0
        for j, n in enumerate(nibs):
            w |= int(n) << (4 * j)
        cleared = w & ((((w & m) + m) | m)) & 0xFFFFFFFF
        want = 0
        for j, n in enumerate(nibs):
            n = 0 if (n & 7) == 0 else int(n)
            want |= n << (4 * j)
        assert cleared == want


def test_nvfp4_product_is_rounded_toward_zero_before_e2m1():
    # the epilogue page's _nvfp4_quant32 forms v * (1/sf) * (1/global) with a
    # round-toward-zero f32 multiply, then rounds to E2M1 (nearest, ties to
    # even).  Groups with a non-trivial global scale put some products within
    # one f32 step above an E2M1 midpoint, where RZ and RN pick different
    # codes; the oracle must take the RZ one.  RZ is formed here from the exact
    # float64 product of the two f32 factors.
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])

    def e2m1(x):
        # nearest magnitude (ties to the even code), saturating at 6; sign in bit 3, none on zero
        a = np.minimum(np.abs(x), 6.0)
        d = np.abs(a[:, None] - mags[None, :])
        best = np.argmin(d, axis=1)  # the lower code of a tie
        nxt = np.minimum(best + 1, 7)
        tie = (best < 7) & (d[np.arange(a.size), nxt] == d[np.arange(a.size), best])
        best = np.where(tie & (best % 2 == 1), best + 1, best)
        return np.where(best == 0, 0, best | np.where(np.signbit(x), 8, 0)).astype(np.uint8)

    r = np.random.default_rng(77)
    differ = 0
    for trial in range(3000):
        gs_inv = np.float32(1.0) / np.float32(r.uniform(0.3, 3.0))
        v = (r.standard_normal(16) * r.uniform(0.5, 20)).astype(np.float32)
        # nudge one element onto a midpoint of the scaled grid
        nib, sfc = oracle.nvfp4_group16(v, float(gs_inv))
        sf = np.float32(oracle.e4m3_decode(sfc))
        rcp = np.float32(np.float32(1.0) / sf) * gs_inv
        mid = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])[r.integers(0, 7)]
        j = int(r.integers(1, 16))
        if abs(v[j]) < np.max(np.abs(v)):
            v[j] = np.float32(mid / np.float64(rcp)) * (1 if r.random() < 0.5 else -1)
            for _ in range(int(r.integers(0, 3))):
                v[j] = np.nextafter(v[j], np.float32(np.inf) * np.sign(v[j]))
        nib, sfc = oracle.nvfp4_group16(v, float(gs_inv))
        sf = np.float32(oracle.e4m3_decode(sfc))
        rcp = np.float32(np.float32(1.0) / sf) * gs_inv
        exact = v.astype(np.float64) * np.float64(rcp)
        rn = exact.astype(np.float32)
        rz = np.where(np.abs(rn.astype(np.float64)) > np.abs(exact), np.nextafter(rn, np.float32(0)), rn)
        want = e2m1(rz.astype(np.float64))
        assert np.array_equal(nib, want), (trial, v, nib, want)
        differ += int(np.sum(e2m1(rn.astype(np.float64)) != want))
    assert differ > 20  # the RZ / RN difference was exercised


# ------------------------------------------------------- norm and rope

def test_head_rmsnorm_unit_rms_with_zero_gamma_and_constant_rows():
    g0 = np.zeros(128, np.uint16)  # bf16 0.0
    for _ in range(20):
        y = (rng.standard_normal(128) * 10 ** rng.uniform(-2, 2)).astype(np.float32)
        z = oracle.head_rmsnorm(y, g0, 1e-6)
        ms = float(np.mean(y.astype(np.float64) ** 2))
        eps = float(np.float32(1e-6))  # eps is an f32 argument
        assert abs(math.sqrt(np.mean(z ** 2)) - math.sqrt(ms / (ms + eps))) < 1e-12
    gam = np.array([oracle.bf16_encode(v) for v in rng.standard_normal(128) * 0.1], np.uint16)
    gd = np.array([oracle.bf16_decode(b) for b in gam])
    z = oracle.head_rmsnorm(np.full(128, -3.0, np.float32), gam, 0.0)
    assert np.allclose(z, -(1.0 + gd), rtol=0, atol=1e-12)


def test_rope_identity_rotation_and_norms():
    z = rng.standard_normal(128)
    tab = workloads.cos_sin_table(4096)
    # position 0: cos = 1, sin = 0 exactly in bf16 -> identity
    assert np.array_equal(oracle.rope_neox(z, tab[0]), z)
    for p in rng.integers(1, 4096, 50):
        out = oracle.rope_neox(z, tab[p])
        assert np.array_equal(out[64:], z[64:])
        c = np.array([oracle.bf16_decode(b) for b in tab[p][:32]])
        s = np.array([oracle.bf16_decode(b) for b in tab[p][32:]])
        n_in = z[:32] ** 2 + z[32:64] ** 2
        n_out = out[:32] ** 2 + out[32:64] ** 2
        assert np.allclose(n_out, n_in * (c ** 2 + s ** 2), rtol=1e-12, atol=1e-12)
        assert np.all(np.abs(c ** 2 + s ** 2 - 1) < 2 ** -6)
    # a quarter turn (cos 0, sin 1): x' = -y, y' = x
    quarter = np.array([oracle.bf16_encode(0.0)] * 32 + [oracle.bf16_encode(1.0)] * 32, np.uint16)
    out = oracle.rope_neox(z, quarter)
    assert np.array_equal(out[:32], -z[32:64]) and np.array_equal(out[32:64], z[:32])


# -------------------------------------------------------------- prologue

def _cfg(H=512, weight_fmt=0, eps=1e-6):
    return oracle.Config(H, 16, 1, 1, 1, weight_fmt, 0, 16, 8, 0, eps)


def test_prologue_residual_matches_torch_f32_sum():
    H = 512
    a = torch.randn(H, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    b = (torch.randn(H, generator=torch.Generator().manual_seed(6)) * 100).to(torch.bfloat16)
    ref = (a.float() + b.float()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ar = a.view(torch.int16).numpy().view(np.uint16)
    res = b.view(torch.int16).numpy().view(np.uint16)
    residual, xq, xs, _ = oracle.prologue_row(_cfg(H), ar, res, np.zeros(H, np.uint16))
    assert np.array_equal(residual, ref)


def test_prologue_per_token_amax_maps_to_448_and_unit_rms():
    H = 512
    for seed in range(5):
        g = torch.Generator().manual_seed(seed)
        ar = workloads._bf16_bits(torch.randn(H, generator=g) * 3)
        res = workloads._bf16_bits(torch.randn(H, generator=g))
        _, xq, xs, _ = oracle.prologue_row(_cfg(H), ar, res, np.zeros(H, np.uint16))
        deq = np.array([oracle.e4m3_decode(c) for c in xq])
        assert np.max(np.abs(deq)) == 448.0
        n = deq * xs
        assert abs(math.sqrt(np.mean(n ** 2)) - 1.0) < 0.03  # gamma = 0 -> unit RMS, FP8 noise
    # a constant row normalises to +-1 * (1 + gamma): every code is +-448
    ar = np.full(H, oracle.bf16_encode(2.0), np.uint16)
    res = np.full(H, oracle.bf16_encode(-0.5), np.uint16)
    _, xq, xs, _ = oracle.prologue_row(_cfg(H, eps=0.0), ar, res, np.zeros(H, np.uint16))
    assert (xq == 0x7E).all() and xs == np.float32(1.0) / np.float32(448.0)


def test_prologue_mx_blocks():
    H = 512
    g = torch.Generator().manual_seed(9)
    ar = workloads._bf16_bits(torch.randn(H, generator=g))
    res = workloads._bf16_bits(torch.randn(H, generator=g) * 4)
    _, xq, _, xsf = oracle.prologue_row(_cfg(H, weight_fmt=1), ar, res, np.zeros(H, np.uint16))
    deq = np.array([oracle.e4m3_decode(c) for c in xq]).reshape(H // 32, 32)
    bmax = np.abs(deq).max(axis=1)
    assert np.all((bmax >= 224.0) & (bmax <= 448.0))  # minimal power of two
    n = deq * np.array([oracle.e8m0_decode(c) for c in xsf])[:, None]
    assert abs(math.sqrt(np.mean(n ** 2)) - 1.0) < 0.03


def _e4m3_torch(x):
    """torch's round-to-nearest-even E4M3 cast (values already within +-448)."""
    t = torch.from_numpy(np.clip(np.asarray(x, np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_midpoint_distance(x):
    """Relative distance of each |x| from the nearest midpoint between two
    neighbouring E4M3 magnitudes (where one rounding step can flip a code)."""
    mags = np.array(sorted({abs(oracle.e4m3_decode(c)) for c in range(0x7F)}), np.float64)
    mids = (mags[1:] + mags[:-1]) / 2
    a = np.abs(np.asarray(x, np.float64))
    return np.min(np.abs(a[:, None] - mids[None, :]), axis=1) / np.maximum(a, 1e-30)


@pytest.mark.parametrize("c,eps", [(0.75, 0.3), (-2.5, 1e-6), (0.0625, 0.01)])
@pytest.mark.parametrize("fmt", [0, 1])
def test_prologue_constant_row_with_gamma_has_its_closed_form(c, eps, fmt):
    # Gemma RMSNorm of a constant row c with per-element gamma (pre_attn page,
    # norm_quant): mean(acc^2) = c^2 exactly, so n_k = c / sqrt(c^2 + eps) *
    # (1 + gamma_k) in closed form.  The per-token scale is max|n| / 448 and the
    # codes are e4m3(n_k / s) = e4m3(448 (1 + gamma_k) sign(c) / max|1 + gamma|).
    # A (1 - gamma) slip, a gamma read at the wrong index, a dropped eps or an
    # H - 1 divisor moves a code or the scale.
    H = 512
    g = torch.Generator().manual_seed(int(abs(c) * 1000) + fmt)
    gam = workloads._bf16_bits(torch.randn(H, generator=g) * 0.3)
    gd = bf16_f64(gam)
    ar = np.full(H, oracle.bf16_encode(c), np.uint16)
    res = np.zeros(H, np.uint16)
    eps32 = float(np.float32(eps))
    n = c / math.sqrt(c * c + eps32) * (1.0 + gd)           # float64 closed form
    _, xq, xs, xsf = oracle.prologue_row(_cfg(H, weight_fmt=fmt, eps=eps), ar, res, gam)
    if fmt == 0:
        s = np.max(np.abs(n)) / 448.0
        assert abs(xs - s) <= 2.0 ** -22 * s, (xs, s)
        q = n / s
    else:
        e = np.array([oracle.mx_exponent(float(np.float32(a))) for a in np.abs(n).reshape(-1, 32).max(axis=1)])
        assert np.array_equal(xsf, (e + 127).astype(np.uint8))
        q = n * np.repeat(2.0 ** -e, 32)
    clear = _e4m3_midpoint_distance(q) > 2.0 ** -18        # no f32 rounding can flip these
    assert clear.mean() > 0.95
    assert np.array_equal(xq[clear], _e4m3_torch(q)[clear])


@pytest.mark.parametrize("H,a,b,eps", [(512, 1.5, -0.25, 1e-6), (6144, 3.0, 0.5, 0.5), (1024, -0.125, 0.0, 0.0),
                                       (6144, 40.0, -7.0, 1e-6)])
def test_prologue_two_valued_row_pins_rstd_to_f32_precision(H, a, b, eps):
    # a row alternating a, b has mean(acc^2) = (a^2 + b^2) / 2 exactly, so
    # rstd = 1 / sqrt((a^2 + b^2) / 2 + eps) and (gamma = 0) the per-token scale
    # is max(|a|, |b|) rstd / 448: checked to f32 precision (an H - 1 divisor is
    # off by 1 / (2H), a dropped eps by eps / mean)
    row = np.array([oracle.bf16_encode(a), oracle.bf16_encode(b)] * (H // 2), np.uint16)
    eps32 = float(np.float32(eps))
    rstd = 1.0 / math.sqrt((a * a + b * b) / 2.0 + eps32)
    s = max(abs(a), abs(b)) * rstd / 448.0
    _, xq, xs, _ = oracle.prologue_row(_cfg(H, eps=eps), np.zeros(H, np.uint16), row, np.zeros(H, np.uint16))
    assert abs(xs - s) <= 2.0 ** -22 * s, (xs, s)
    q = np.array([a, b] * (H // 2)) * rstd / s
    clear = _e4m3_midpoint_distance(q) > 2.0 ** -18
    assert np.array_equal(xq[clear], _e4m3_torch(q)[clear])


def bf16_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_torch(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("cache", ["fp8", "nvfp4"])
def test_step_q_and_index_q_heads_are_norm_rope_of_their_own_slice(cache):
    # q heads (epilogue page, q branch): bf16(z) and e4m3(z * (1 / q_fp8_scale))
    # with z = RoPE(RMSNorm(y_head, g_q)); index_q heads: bf16(z) and e4m3(z)
    # with g_iq (pre_attn page head tasks; epilogue page index_q branch).  Each
    # head is checked against the pinned norm and RoPE of its own slice of the
    # projection, and the E4M3 / bf16 roundings against torch's casts.  A g_q /
    # g_iq swap, q without RoPE, q_fp8 times the scale instead of divided by
    # it, or a head written at another head's offset fails here.
    wl = workloads.tiny().replace(name=f"qpin_{cache}", nkv=2, n_q=0, n_iq=0, M=3, q_fp8=True, iq_fp8=True,
                                  q_fp8_scale=0.37, cache_fmt=cache, pool_pages=64,
                                  weight_fmt="ptpc" if cache == "fp8" else "mx")
    st = workloads.host_state(wl)
    y = oracle.run_rows(wl, st, range(wl.M), want_y=True)
    inv = np.float32(1.0) / np.float32(wl.q_fp8_scale)
    iq0 = wl.n_q + 2 * wl.nkv
    assert not np.array_equal(st["g_q"], st["g_iq"])
    for m in range(wl.M):
        cs = st["cos_sin"][st["positions"][m]]
        for j in range(wl.n_q):
            z = np.float32(oracle.rope_neox(oracle.head_rmsnorm(y[m, j * 128:(j + 1) * 128], st["g_q"], wl.eps), cs))
            sl = slice(j * 128, (j + 1) * 128)
            assert np.array_equal(st["q_bf16"][m, sl], _bf16_torch(z)), (m, j)
            assert np.array_equal(st["q_fp8"][m, sl], _e4m3_torch(z * inv)), (m, j)
        for j in range(wl.n_iq):
            h = iq0 + j
            z = np.float32(oracle.rope_neox(oracle.head_rmsnorm(y[m, h * 128:(h + 1) * 128], st["g_iq"], wl.eps), cs))
            sl = slice(j * 128, (j + 1) * 128)
            assert np.array_equal(st["iq_bf16"][m, sl], _bf16_torch(z)), (m, j)
            assert np.array_equal(st["iq_fp8"][m, sl], _e4m3_torch(z)), (m, j)


# ------------------------------------------------------------ projection

@pytest.mark.parametrize("fmt", ["ptpc", "mx"])
def test_projection_equals_numpy_matmul_of_dequantised_operands(fmt):
    wl = workloads.tiny().replace(weight_fmt=fmt, M=3)
    st = workloads.host_state(wl)
    cfg = oracle.oracle_config(wl)
    lut = np.array([oracle.e4m3_decode(c) for c in range(256)], np.float64)
    lut[np.isnan(lut)] = 0
    W = lut[st["w"]]
    if fmt == "ptpc":
        W = W * st["w_scale"].astype(np.float64)[:, None]
    else:
        W = W * np.repeat(2.0 ** (st["wsf"].astype(np.float64) - 127), 32, axis=1)
    for m in range(wl.M):
        _, xq, xs, xsf = oracle.prologue_row(cfg, st["ar"][m], st["res"][m], st["g_in"])
        x = lut[xq] * (xs if fmt == "ptpc" else np.repeat(2.0 ** (xsf.astype(np.float64) - 127), 32))
        ref = W @ x
        y = oracle.project_row(cfg, xq, xs, xsf if fmt == "mx" else None, st["w"],
                               st.get("w_scale"), st.get("wsf"))
        assert np.allclose(y, ref, rtol=1e-6, atol=1e-6)


# ----------------------------------------------------------------- layouts

def _load_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append([int(v) for v in line.split()])
    return rows


def test_layout_offsets_match_values_worked_from_the_pages():
    L = oracle.lib()
    for kind, *args, want in _load_golden("layout_offsets.txt"):
        if kind == 0:    # fp8 K shuffle: page16, h, nkv, t, d
            got = L.ora_fp8_k_offset(*args)
        elif kind == 1:  # fp8 V: page16, h, nkv, t, d
            got = L.ora_fp8_v_offset(*args)
        elif kind == 2:  # nvfp4 V-swizzled scale: bs, slot, t, g
            got = L.ora_nvfp4_sf_vswz_offset(*args)
        elif kind == 3:  # nvfp4 linear scale: bs, slot, t, g
            got = L.ora_nvfp4_sf_linear_offset(*args)
        elif kind == 4:  # nvfp4 data byte: bs, slot, t, d
            got = L.ora_nvfp4_data_offset(*args)
        elif kind == 5:  # page16_of: slot, kps
            got = L.ora_page16_of(*args)
        elif kind == 6:  # F8_128x4: r, kb, ksf
            got = L.ora_sf128x4_offset(*args)
        assert got == want, (kind, args, got, want)


def _cute_offset(coord_shape_stride):
    """Evaluate a CuTe layout (shape, stride) at a flat-per-mode coordinate."""
    off = 0
    for idx, shape, stride in coord_shape_stride:
        if isinstance(shape, tuple):
            for s, d in zip(shape, stride):
                off += (idx % s) * d
                idx //= s
        else:
            off += idx * stride
    return off


@pytest.mark.parametrize("bs", [4, 16, 32])
def test_nvfp4_views_agree_with_the_pages_cute_layouts(bs):
    L = oracle.lib()
    slot_bytes = bs * 72
    for s in range(3):
        for t in range(bs):
            for g in range(8):
                # vsf: ((2,4),(4,bs//4),nslots) : ((4,8),(1,32),slot_bytes) + sf_off
                want = bs * 64 + _cute_offset([(g, (2, 4), (4, 8)), (t, (4, bs // 4), (1, 32)),
                                               (s, 0, slot_bytes)])
                assert L.ora_nvfp4_sf_vswz_offset(bs, s, t, g) == want
                # sf: (8, bs, nslots) : (1, 8, slot_bytes) + sf_off
                want = bs * 64 + g + 8 * t + s * slot_bytes
                assert L.ora_nvfp4_sf_linear_offset(bs, s, t, g) == want
            for d in range(0, 128, 2):
                # data as bytes: (32, 2, bs, nslots) : (1, 32, 64, slot_bytes)
                want = _cute_offset([((d % 64) // 2, 0, 1), (d // 64, 0, 32), (t, 0, 64), (s, 0, slot_bytes)])
                assert L.ora_nvfp4_data_offset(bs, s, t, d) == want


def test_sf128x4_pack_matches_the_pages_permutation():
    for R, ksf in ((128, 4), (256, 16), (300, 8), (9856, 192)):
        src = rng.integers(0, 255, (R, ksf)).astype(np.uint8)
        got = oracle.pack_sf128x4(src, pad=0)
        rp = (R + 127) // 128 * 128
        pad = np.zeros((rp, ksf), np.uint8)
        pad[:R] = src
        # [R/128, Ksf/4, 32, 4, 4]: (row block, k quad, row % 32, (row % 128) / 32, k % 4)
        want = pad.reshape(rp // 128, 4, 32, ksf // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
        assert np.array_equal(got, want)


# --------------------------------------------------------- the whole step

def _dequant_fp8_k_token(st, wl, slot, h):
    p16, t = slot // 16, slot % 16
    page = st["k_cache"].reshape(-1, wl.nkv, 2048)[p16, h]
    codes = page.reshape(8, 16, 16)[:, t, :].reshape(128)  # [d/16][t][d%16]
    return codes


def test_step_fp8_caches_touch_only_the_slots_and_decode_consistently():
    wl = workloads.tiny().replace(q_fp8=True, iq_fp8=True, skip_rows=(2,))
    st = workloads.host_state(wl)
    y = oracle.run_rows(wl, st, range(wl.M), want_y=True)
    fresh = workloads.host_state(wl)
    touched_pages = set()
    for m in range(wl.M):
        slot = int(st["slot_mapping"][m])
        if slot < 0:
            continue
        touched_pages.add(slot // 16)
    # untouched pages keep the sentinel
    kc = st["k_cache"].reshape(-1, wl.nkv, 2048)
    for p in range(wl.num_pages16):
        if p not in touched_pages:
            assert (kc[p] == workloads.SENTINEL).all()
    for m in range(wl.M):
        slot = int(st["slot_mapping"][m])
        if slot < 0:
            continue
        p16, t = slot // 16, slot % 16
        # V codes sit transposed ([d][t]); dequantised they match the raw projection
        vpage = st["v_cache"].reshape(-1, wl.nkv, 2048)[p16, 0].reshape(128, 16)
        vs = st["v_scale"].reshape(-1, wl.nkv, 16)[p16, 0, t]
        v = y[m, (wl.n_q + wl.nkv) * 128:(wl.n_q + wl.nkv + 1) * 128]
        deq = np.array([oracle.e4m3_decode(c) for c in vpage[:, t]]) * vs
        assert np.allclose(deq, v, rtol=2 ** -3, atol=vs * 2 ** -8)
        assert abs(np.max(np.abs(v)) / 448.0 - vs) <= 1e-6 * vs
        # K codes in the shuffle order decode to bf16(norm + rope of k) / ks
        kcodes = _dequant_fp8_k_token(st, wl, slot, 0)
        ks = st["k_scale"].reshape(-1, wl.nkv, 16)[p16, 0, t]
        assert max(abs(oracle.e4m3_decode(c)) for c in kcodes) == 448.0
        # the k head's q-like output is not written anywhere else: compare
        # against norm + rope recomputed from y
        k = y[m, wl.n_q * 128:(wl.n_q + 1) * 128]
        z = oracle.rope_neox(oracle.head_rmsnorm(k, st["g_k"], wl.eps), st["cos_sin"][st["positions"][m]])
        deq = np.array([oracle.e4m3_decode(c) for c in kcodes]) * ks
        assert np.allclose(deq, z, rtol=2 ** -3, atol=ks * 2 ** -8)
        # exactly (pre_attn page, head tasks: the K store quantises the
        # bf16-rounded normed + roped value by the scale of its f32 amax):
        # e4m3(f32(bf16(z)) / ks), ks = f32(amax(f32(z)) / 448)
        zf = np.float32(z)
        ks_want = np.float32(np.max(np.abs(zf))) / np.float32(448.0)
        assert ks == ks_want
        zb = torch.from_numpy(zf).to(torch.bfloat16).to(torch.float32).numpy()
        assert np.array_equal(kcodes, _e4m3_torch(zb / ks_want))
        # the index cache row holds e4m3(bf16(index_k))
        ik = y[m, (wl.n_heads - 1) * 128:]
        z = oracle.rope_neox(oracle.head_rmsnorm(ik, st["g_ik"], wl.eps), st["cos_sin"][st["positions"][m]])
        row = st["index_cache"].reshape(-1, 128)[slot]
        assert np.allclose([oracle.e4m3_decode(c) for c in row], z, rtol=2 ** -3, atol=2 ** -9)
    # the skipped row wrote no cache byte but still wrote q
    assert (st["q_bf16"][2] != 0xA5A5).all()
    # q_fp8 and q_bf16 agree within FP8 precision
    qb = np.array([oracle.bf16_decode(b) for b in st["q_bf16"].reshape(-1)])
    qf = np.array([oracle.e4m3_decode(c) for c in st["q_fp8"].reshape(-1)])
    assert np.allclose(qf, qb, rtol=2 ** -4, atol=2 ** -9)
    assert not np.array_equal(fresh["k_cache"], st["k_cache"])


def test_step_nvfp4_caches_decode_consistently():
    wl = workloads.Workload("t4", H=512, nkv=2, M=6, weight_fmt="mx", cache_fmt="nvfp4", seed=7,
                            positions="uniform", max_pos=512, pool_pages=32, q_fp8=True,
                            iq_fp8=True, page_pad=64, k_global=0.5, v_global=2.0)
    st = workloads.host_state(wl)
    y = oracle.run_rows(wl, st, range(wl.M), want_y=True)
    bs = wl.block_size
    for m in range(wl.M):
        slot = int(st["slot_mapping"][m])
        page = st["kv_cache"].reshape(wl.kv_pages, wl.kv_page_bytes)[slot // bs]
        t = slot % bs
        for h in range(wl.nkv):
            for role, gsc in (("k", wl.k_global), ("v", wl.v_global)):
                sl = 2 * h + (role == "v")
                blk = page[sl * bs * 72:(sl + 1) * bs * 72]
                data = blk[:bs * 64].reshape(bs, 2, 32)[t].reshape(64)
                nib = np.stack([data & 15, data >> 4], axis=1).reshape(128)  # even element low
                sfb = blk[bs * 64:].reshape(bs // 4, 8, 4) if role == "v" else blk[bs * 64:].reshape(bs, 8)
                if role == "v":  # byte g of token t at (t/4*4 + g/2)*8 + g%2*4 + t%4
                    sfs = [blk[bs * 64 + ((t // 4) * 4 + g // 2) * 8 + (g % 2) * 4 + t % 4] for g in range(8)]
                else:
                    sfs = list(sfb[t])
                deq = np.array([oracle.e2m1_decode(n) for n in nib]) * np.repeat(
                    [oracle.e4m3_decode(s) for s in sfs], 16) * gsc
                if role == "v":
                    ref = y[m, (wl.n_q + wl.nkv + h) * 128:(wl.n_q + wl.nkv + h + 1) * 128]
                else:
                    k = y[m, (wl.n_q + h) * 128:(wl.n_q + h + 1) * 128]
                    ref = oracle.rope_neox(oracle.head_rmsnorm(k, st["g_k"], wl.eps),
                                           st["cos_sin"][st["positions"][m]])
                gmax = np.abs(ref).reshape(8, 16).max(axis=1)
                tol = np.repeat(gmax, 16) / 6 * 1.07 + 1e-6
                assert np.all(np.abs(deq - ref) <= tol), (m, h, role)


# --------------------------------------------------------- indexer scores

def test_index_scale_is_the_attention_scale_times_log2e():
    # exp2 of the scaled score is exp of sm_scale * q.k: 2^(x log2 e) = e^x
    for s in (1.0, 128 ** -0.5, 0.03):
        v = oracle.index_scale_log2e(s)
        assert abs(v - s * 1.4426950408889634) <= 1e-15 * v
        assert abs(2.0 ** v - math.e ** s) <= 1e-14 * math.e ** s


def _one_request(seq_len, q_len, bt_width, seed):
    g = np.random.default_rng(seed)
    nb = (seq_len + 127) // 128
    bt = np.full((1, bt_width), -1, np.int32)
    bt[0, :nb] = g.permutation(nb + 5)[:nb]
    iq = workloads._bf16_bits(torch.randn(q_len, 128, generator=torch.Generator().manual_seed(seed)))
    keys = workloads._e4m3_bits(torch.randn((nb + 5) * 128, 128, generator=torch.Generator().manual_seed(seed + 1)))
    return iq, keys, bt, np.array([seq_len], np.int32)


def test_index_score_masks_match_the_hand_worked_patterns():
    rows = _load_golden("index_masks.txt")
    for seq_len, q_len, init, local, i, lo, hi, written in rows:
        iq, keys, bt, sl = _one_request(seq_len, q_len, 16, seq_len)
        out = oracle.index_scores(iq, keys, bt, sl, q_len, init, local, 0.5, 16 * 128)[i]
        finite = np.isfinite(out)
        assert np.array_equal(np.nonzero(finite)[0], np.arange(lo, hi)), (seq_len, q_len, init, local, i)
        assert np.all(np.isneginf(out[:written][~finite[:written]]))
        assert np.all(np.isnan(out[written:]))


def test_index_scores_equal_a_float64_dot_product_of_the_dequantised_rows():
    iw = workloads.IndexWorkload("pin", R=3, q_len=3, seq_lo=130, seq_hi=900, bt_width=8, seed=11, n_iq=2, head=1)
    st = workloads.index_host_state(iw)
    scale = float(np.float32(oracle.index_scale_log2e(iw.sm_scale)))
    iq = st["iq"][:, 128:256]  # head 1 of each row
    out = oracle.index_scores(iq, st["index_cache"], st["block_table"], st["seq_lens"], iw.q_len, 1, 1,
                              scale, 8 * 128)
    lut = np.array([oracle.e4m3_decode(c) for c in range(256)], np.float64)
    keys = lut[st["index_cache"].reshape(-1, 128)]
    qf = (iq.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    checked = 0
    for m in range(iw.M):
        r, i = divmod(m, iw.q_len)
        p = int(st["seq_lens"][r]) - iw.q_len + i
        for j in np.nonzero(np.isfinite(out[m]))[0]:
            slot = int(st["block_table"][r, j // 128]) * 128 + j % 128
            want = np.float32(np.dot(qf[m], keys[slot]) * scale)
            assert j <= p
            assert abs(float(out[m, j]) - float(want)) <= abs(float(want)) * 2.0 ** -23, (m, j)
            checked += 1
    assert checked > 1000
