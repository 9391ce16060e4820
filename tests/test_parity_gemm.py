"""GPU parity of the tensor-core path (prologue + persistent tcgen05 GEMM with
the fused head epilogue) against the CPU oracle, through the C-ABI.  Every
case compares every row (the oracle runs its independent rows on all host
cores) and checks that no byte outside the written slots changed."""

import numpy as np
import pytest

import workloads
from tests import harness

pytestmark = pytest.mark.gpu


def _flags(force_gemm=True, tiles=None):
    from indexer_projection_gb300 import binding as B
    f = B.PA_FLAG_FORCE_GEMM if force_gemm else 0
    if tiles == "single":
        f |= B.PA_FLAG_GEMM_SINGLE
    elif tiles == "pair":
        f |= B.PA_FLAG_GEMM_PAIR
    return f


def check(wl, rows=None, flags=None, gemm_grid=0):
    st = workloads.host_state(wl)
    g = harness.GpuRun(wl, st, flags=_flags() if flags is None else flags, gemm_grid=gemm_grid)
    g.run()
    got = g.results()
    if rows is None:
        rows = list(range(wl.M))
    ref = harness.oracle_run(wl, st, rows)
    tally = harness.compare(wl, got, ref, rows, all_rows=range(wl.M))
    assert g.runner.device_status() == 0
    return tally


def small(name, M, fmt="ptpc", cache="fp8", nkv=1, H=512, seed=21, **kw):
    base = dict(positions="uniform", max_pos=4096, pool_pages16=2048, pool_pages=512, q_fp8=True, iq_fp8=True)
    base.update(kw)
    return workloads.Workload(name, H=H, nkv=nkv, M=M, weight_fmt=fmt, cache_fmt=cache, seed=seed, **base)


TILES = ["single", "pair"]


@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("fmt", ["ptpc", "mx"])
@pytest.mark.parametrize("cache", ["fp8", "nvfp4"])
def test_small_ragged(fmt, cache, tiles):
    # nkv = 2: 39 heads, so the pair kernel's last tile has a zero-filled second head
    check(small(f"g_{fmt}_{cache}_{tiles}", 200, fmt, cache, nkv=2, skip_rows=(3, 130)), flags=_flags(tiles=tiles))


@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("M", [1, 5, 17, 127, 128, 129, 256, 300])
def test_token_counts(M, tiles):
    check(small(f"g_m{M}_{tiles}", M, "mx", "nvfp4", H=1024, seed=M), flags=_flags(tiles=tiles))


@pytest.mark.parametrize("tiles,grid", [("single", 1), ("single", 3), ("single", 37), ("pair", 2), ("pair", 6),
                                        ("pair", 38)])
def test_persistent_grid_override(tiles, grid):
    # fewer CTAs than tiles: every CTA (pair) walks many tiles
    check(small(f"g_grid{grid}_{tiles}", 600, "mx", "fp8", nkv=1, H=768, seed=grid), flags=_flags(tiles=tiles),
          gemm_grid=grid)


@pytest.mark.parametrize("tiles", TILES)
def test_per_channel_nvfp4_ragged_pair_rows(tiles):
    check(small(f"g_pc_{tiles}", 389, "ptpc", "nvfp4", nkv=4, H=640, seed=3, page_pad=32, k_global=0.7,
                v_global=1.3), flags=_flags(tiles=tiles))


@pytest.mark.parametrize("tiles", TILES)
def test_long_k_and_outliers(tiles):
    check(small(f"g_k6144_{tiles}", 136, "ptpc", "fp8", nkv=1, H=6144, seed=8, outlier_frac=0.05),
          flags=_flags(tiles=tiles))


@pytest.mark.parametrize("tiles", TILES)
def test_skipped_slots_static_scale_separate_index_slots(tiles):
    # skipped rows scattered over several warps (the V rows leave a warp at a
    # time, so a warp mixes rows with and without a slot), K / V scales fixed
    # at 1, index_k rows in their own slots
    check(small(f"g_skip_{tiles}", 200, "ptpc", "fp8", nkv=2, seed=31, skip_rows=(0, 5, 6, 37, 64, 130, 199),
                static_kv_scale=True, separate_index_slots=True), flags=_flags(tiles=tiles))


@pytest.mark.parametrize("tiles", TILES)
def test_kv_page_stride_16(tiles):
    wl = small(f"g_kps16_{tiles}", 150, "mx", "fp8", nkv=2, seed=32, kv_page_stride=16, pool_pages16=256)
    st = workloads.host_state(wl)
    # distinct slots below 128 * 16, so page16 ids stay below 256
    st["slot_mapping"] = np.random.default_rng(32).permutation(128 * 16)[:wl.M].astype(np.int64)
    g = harness.GpuRun(wl, st, flags=_flags(tiles=tiles))
    g.run()
    ref = harness.oracle_run(wl, st, range(wl.M))
    harness.compare(wl, g.results(), ref, range(wl.M))
    assert g.runner.device_status() == 0


@pytest.mark.parametrize("tiles", TILES)
def test_out_of_range_slots_are_flagged_not_written(tiles):
    from indexer_projection_gb300 import binding as B
    wl = small(f"g_oor_{tiles}", 140, "ptpc", "fp8", nkv=2, seed=33)
    st = workloads.host_state(wl)
    bad = (1, 40, 139)
    for m in bad:
        st["slot_mapping"][m] = wl.num_pages16 * 16 + 5 + m  # beyond the cache
        st["index_slot_mapping"][m] = wl.num_index_slots + 9 + m
    g = harness.GpuRun(wl, st, flags=_flags(tiles=tiles))
    g.run()
    got = g.results()
    assert g.runner.device_status() == B.PA_DEV_SLOT_RANGE
    ok_rows = [m for m in range(wl.M) if m not in bad]
    ref = harness.oracle_run(wl, st, ok_rows)
    harness.compare(wl, got, ref, ok_rows, all_rows=ok_rows)


def test_spec_decode_config():
    check(workloads.spec_decode(), flags=0)


@pytest.mark.parametrize("tiles", [None, "single"])
def test_configs_head_layout_with_twice_the_index_q_heads(tiles):
    # the configs' N for nkv = 2 and 4 (5248, 10368) is the layout with
    # 2 * nkv index_q heads (41 and 81 heads, odd: the pair kernel's last tile
    # has a zero-filled second head)
    check(workloads.spec_decode().replace(n_iq=4), flags=_flags(force_gemm=False, tiles=tiles))
    check(workloads.prefill().replace(n_iq=8, M=1024, requests=1, q_len=1024),
          flags=_flags(force_gemm=False, tiles=tiles))


@pytest.mark.parametrize("tiles", [None, "single"])
def test_prefill_config(tiles):
    check(workloads.prefill(), flags=_flags(force_gemm=False, tiles=tiles))


@pytest.mark.parametrize("M", [64, 256, 1024, 4096, 16384])
def test_sweep_config_tensor_core_points(M):
    check(workloads.sweep(M), flags=0)


def test_path_choice():
    from indexer_projection_gb300 import binding as B
    from indexer_projection_gb300.runner import PreAttn

    def path(M, flags=0, nkv=4):
        r = PreAttn(6144, nkv, weight_format=B.PA_WEIGHT_MXFP8, cache_format=B.PA_CACHE_FP8, max_tokens=16384,
                    flags=flags)
        return B.pre_attn_path(r.handle, M)

    skinny = (B.PA_PATH_GEMV, B.PA_PATH_GEMV_FUSED, B.PA_PATH_GEMV_PERSIST)
    assert path(8) in skinny and path(16) in skinny
    # 77 heads at nkv = 4: more than two waves of 16-CTA clusters on 152 SMs;
    # 20 heads at nkv = 1 (the decode shape) stay on the one-cluster-a-head grid
    assert path(8) == B.PA_PATH_GEMV_PERSIST and path(8, B.PA_FLAG_FUSE) == B.PA_PATH_GEMV_FUSED
    assert path(8, nkv=1) == B.PA_PATH_GEMV
    assert path(8, B.PA_FLAG_GEMV_REGULAR) == B.PA_PATH_GEMV
    assert path(8, B.PA_FLAG_GEMV_PERSIST, nkv=1) == B.PA_PATH_GEMV_PERSIST
    assert path(8, B.PA_FLAG_FORCE_GEMM) in (B.PA_PATH_GEMM_SINGLE, B.PA_PATH_GEMM_PAIR)
    assert path(8192) == B.PA_PATH_GEMM_PAIR  # 1312 pair tiles vs 5184 single tiles
    assert path(8192, B.PA_FLAG_GEMM_SINGLE) == B.PA_PATH_GEMM_SINGLE
    assert path(64, B.PA_FLAG_GEMM_PAIR) == B.PA_PATH_GEMM_PAIR
    assert path(17) in (B.PA_PATH_GEMM_SINGLE, B.PA_PATH_GEMM_PAIR)


@pytest.mark.parametrize("fmt", ["ptpc", "mx"])
def test_prologue_fast_path_is_bitwise_the_exact_path(fmt):
    # the many-row prologue quantises from a cheap normalised value where
    # every value within 2^-20 of it gives the same code and scale, and from
    # the exact one elsewhere: forcing the exact path everywhere must change
    # no output bit (outlier rows push many values near code boundaries)
    from indexer_projection_gb300 import binding as B
    wl = small("fastpath", 2048, fmt=fmt, H=6144, nkv=1, seed=71, outlier_frac=0.05)
    st = workloads.host_state(wl)
    outs = []
    for extra in (0, B.PA_FLAG_EXACT_NORM):
        g = harness.GpuRun(wl, st, flags=_flags() | extra)
        g.run()
        outs.append(g.results())
        assert g.runner.device_status() == 0
    for k in outs[0]:
        assert np.array_equal(outs[0][k], outs[1][k]), k
