"""GPU parity of the skinny-M path (M <= 16: prologue + weight-streaming GEMV
+ last-arriver head epilogue) against the CPU oracle, through the C-ABI."""

import numpy as np
import pytest

import workloads
from tests import harness

pytestmark = pytest.mark.gpu


def _gemv_flags():
    from indexer_projection_gb300 import binding as B
    return B.PA_FLAG_FORCE_GEMV


def check(wl, flags=None, rows=None, runs=1):
    st = workloads.host_state(wl)
    g = harness.GpuRun(wl, st, flags=_gemv_flags() if flags is None else flags)
    for _ in range(runs):
        g.run()
    got = g.results()
    rows = list(range(wl.M)) if rows is None else rows
    ref = harness.oracle_run(wl, st, rows)
    harness.compare(wl, got, ref, rows, all_rows=range(wl.M))
    assert g.runner.device_status() == 0
    return g


def test_tiny():
    check(workloads.tiny())


def test_decode():
    check(workloads.decode())


def test_decode_every_output_and_nvfp4_mx():
    check(workloads.decode().replace(q_fp8=True, iq_fp8=True, q_fp8_scale=0.37))
    check(workloads.decode().replace(weight_fmt="mx", cache_fmt="nvfp4", pool_pages=4096, q_fp8=True,
                                     iq_fp8=True, k_global=0.5, v_global=3.0))


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 9, 13, 16])
def test_token_counts(M):
    check(workloads.tiny().replace(M=M, q_fp8=True, iq_fp8=True))


@pytest.mark.parametrize("nkv", [2, 4])
@pytest.mark.parametrize("fmt", ["ptpc", "mx"])
def test_kv_heads_and_formats(nkv, fmt):
    check(workloads.tiny().replace(nkv=nkv, n_q=0, n_iq=0, weight_fmt=fmt, M=7, iq_fp8=True))


def test_skipped_slots_static_scale_separate_index_slots():
    check(workloads.tiny().replace(M=8, skip_rows=(0, 5), static_kv_scale=True, separate_index_slots=True))


def test_nvfp4_block_sizes_and_page_padding():
    for bs, pad in ((16, 0), (4, 32), (32, 96)):
        check(workloads.Workload(f"nv_bs{bs}", H=512, nkv=2, M=9, weight_fmt="ptpc", cache_fmt="nvfp4",
                                 seed=11 + bs, positions="uniform", max_pos=300, pool_pages=40, block_size=bs,
                                 page_pad=pad, q_fp8=True, iq_fp8=True, skip_rows=(3,)))


def test_outlier_rows_and_custom_heads():
    check(workloads.Workload("odd", H=1024, nkv=2, n_q=8, n_iq=3, M=12, weight_fmt="mx", cache_fmt="fp8",
                             seed=5, positions="uniform", max_pos=1000, pool_pages16=128, outlier_frac=0.2,
                             q_fp8=True, iq_fp8=True))


def test_kv_page_stride_16():
    wl = workloads.tiny().replace(M=6, kv_page_stride=16, pool_pages16=128)
    st = workloads.host_state(wl)
    st["slot_mapping"] = st["slot_mapping"] % (64 * 16)  # page16 ids stay below 128
    g = harness.GpuRun(wl, st, flags=_gemv_flags())
    g.run()
    ref = harness.oracle_run(wl, st, range(wl.M))
    harness.compare(wl, g.results(), ref, range(wl.M))


def test_repeated_calls_reuse_the_workspace():
    # the per-head arrival counters must be back at zero after every call
    check(workloads.decode(), runs=3)


def test_out_of_range_slots_and_positions_are_flagged_not_written():
    from indexer_projection_gb300 import binding as B
    wl = workloads.tiny().replace(M=4)
    st = workloads.host_state(wl)
    st["slot_mapping"][1] = wl.num_pages16 * 16 + 5      # beyond the cache
    st["index_slot_mapping"][1] = wl.num_index_slots + 9
    g = harness.GpuRun(wl, st, flags=_gemv_flags())
    g.run()
    got = g.results()
    assert g.runner.device_status() == B.PA_DEV_SLOT_RANGE
    ok_rows = [0, 2, 3]
    ref = harness.oracle_run(wl, st, ok_rows)
    harness.compare(wl, got, ref, ok_rows, all_rows=ok_rows)
    st2 = workloads.host_state(wl)
    st2["positions"][2] = wl.max_pos + 100
    g2 = harness.GpuRun(wl, st2, flags=_gemv_flags())
    g2.run()
    g2.results()
    assert g2.runner.device_status() == B.PA_DEV_POS_RANGE


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_sweep_config_skinny_points(M):
    check(workloads.sweep(M), flags=0)


@pytest.mark.parametrize("fmt", ["ptpc", "mx"])
def test_persistent_gemv(fmt):
    # the persistent GEMV: resident clusters walk the heads c, c + G, ...
    # with weight buffers and tensor-memory accumulators double-buffered
    from indexer_projection_gb300 import binding as B
    flags = B.PA_FLAG_FORCE_GEMV | B.PA_FLAG_GEMV_PERSIST

    def run(wl, runs=1):
        g = check(wl, flags=flags, runs=runs)
        assert B.pre_attn_path(g.runner.handle, wl.M) == B.PA_PATH_GEMV_PERSIST

    # 77 heads: every cluster takes several, both buffers turn over many times;
    # repeated calls reuse the barriers' fresh state each launch
    run(workloads.sweep(16).replace(name=f"pg77_{fmt}", weight_fmt=fmt, M=16), runs=2)
    run(workloads.sweep(1).replace(name=f"pg77m1_{fmt}", weight_fmt=fmt, cache_fmt="nvfp4", pool_pages=4096))
    run(workloads.decode().replace(weight_fmt=fmt, q_fp8=True, iq_fp8=True))
    # empty K ranges (512: 4 of 16 ranges hold a chunk), fewer heads than clusters
    run(workloads.tiny().replace(M=5, weight_fmt=fmt, q_fp8=True, iq_fp8=True))
    # ragged K: 4352 = 16 ranges of 384 with the last ones short or empty
    run(workloads.Workload(f"pg_ragged_{fmt}", H=4352, nkv=2, M=9, weight_fmt=fmt, cache_fmt="nvfp4", seed=97,
                           positions="uniform", max_pos=500, pool_pages=64, q_fp8=True, iq_fp8=True,
                           outlier_frac=0.2, skip_rows=(3,)))


@pytest.mark.parametrize("H", [128, 2048, 2176, 4352, 16384])
@pytest.mark.parametrize("fmt", ["ptpc", "mx"])
def test_k_ranges(H, fmt):
    # each head's cluster splits K into 8 ranges of ceil(H / 8) rounded up to
    # 64 bytes: empty ranges (H = 128), a ragged last range (2176, 4352) and
    # ranges longer than the registers hold (16384: the units are refilled)
    check(workloads.Workload(f"ks{H}", H=H, nkv=1, M=11 if fmt == "mx" else 5, weight_fmt=fmt, cache_fmt="fp8",
                             seed=H + (fmt == "mx"), positions="uniform", max_pos=500, pool_pages16=64,
                             q_fp8=True, iq_fp8=True))


@pytest.mark.parametrize("fmt", ["ptpc", "mx"])
def test_fused_single_kernel(fmt):
    # the skinny path in one kernel: the row normalisation runs inside the
    # GEMV's clusters (norm partials exchanged among the 16 K ranges)
    from indexer_projection_gb300 import binding as B
    flags = B.PA_FLAG_FORCE_GEMV | B.PA_FLAG_FUSE
    check(workloads.decode().replace(weight_fmt=fmt, q_fp8=True, iq_fp8=True), flags=flags)
    check(workloads.tiny().replace(M=13, nkv=2, n_q=0, n_iq=0, weight_fmt=fmt, iq_fp8=True), flags=flags)
    check(workloads.Workload("fz_ragged", H=4352, nkv=1, M=16, weight_fmt=fmt, cache_fmt="nvfp4", seed=91,
                             positions="uniform", max_pos=500, pool_pages=64, q_fp8=True, iq_fp8=True,
                             outlier_frac=0.2), flags=flags)
    check(workloads.Workload("fz_one", H=6144, nkv=2, M=1, weight_fmt=fmt, cache_fmt="fp8", seed=92,
                             positions="uniform", max_pos=500, pool_pages16=64), flags=flags)


@pytest.mark.parametrize("fmt,H,M,seed", [("ptpc", 6144, 8, 91), ("ptpc", 4352, 3, 92), ("ptpc", 512, 4, 93),
                                          ("ptpc", 6144, 16, 96), ("mx", 6144, 16, 94), ("mx", 512, 5, 95)])
def test_skinny_prologue_codes_and_scales_are_the_oracles(fmt, H, M, seed):
    # White box.  The skinny path's prologue leaves in the workspace the
    # per-token scales at byte 256 (per-channel format) and the FP8 codes
    # [M, H] at the next 256-byte boundary (after the MXFP8 scale atoms,
    # F8_128x4 over M rounded up to 128).  The per-channel scale comes from
    # one exchange (max |acc (1 + gamma)| times rstd, rounded once), not from
    # a pass over the normalised row: every scale and every code must still
    # be the oracle's.  A third of the rows are outliers (x50).
    import oracle
    wl = workloads.Workload(f"pq{H}", H=H, nkv=1, M=M, weight_fmt=fmt, cache_fmt="fp8", seed=seed,
                            outlier_frac=0.3, max_pos=4096, pool_pages16=2048)
    st = workloads.host_state(wl)
    g = harness.GpuRun(wl, st, flags=_gemv_flags())
    g.run()
    assert g.runner.device_status() == 0
    ws = g.runner.workspace.cpu().numpy()

    def up(x):
        return (x + 255) // 256 * 256
    ksf = H // 32
    xs_off = 256
    xsf_off = up(xs_off + 4 * M)
    xq_off = xsf_off + (up((M + 127) // 128 * 128 * ksf) if fmt == "mx" else 0)
    cfg = oracle.oracle_config(wl)
    ref = [oracle.prologue_row(cfg, st["ar"][m], st["res"][m], st["g_in"]) for m in range(M)]
    xq = ws[xq_off:xq_off + M * H].reshape(M, H)
    for m in range(M):
        assert np.array_equal(xq[m], ref[m][1]), m
    if fmt == "ptpc":
        xs = ws[xs_off:xs_off + 4 * M].view(np.float32)
        assert np.array_equal(xs, np.array([r[2] for r in ref], np.float32))
    else:
        rows = np.stack([r[3] for r in ref])
        got = ws[xsf_off:xsf_off + (M + 127) // 128 * 128 * ksf]
        want = oracle.pack_sf128x4(rows, pad=0)
        real = oracle.pack_sf128x4(np.ones_like(rows), pad=0) == 1
        assert np.array_equal(got[real], want[real])
