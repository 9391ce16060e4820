"""GPU parity of the indexer scores (pre_attn_index_scores) against the CPU
oracle, through the C-ABI.

Tolerance: the kernel multiplies bf16 index_q by E4M3 keys exactly and sums
the 128 products in f32, then scales: its error is at most about
128 * 2^-24 of the sum of |products|, so each score must satisfy
|gpu - oracle| <= 2^-16 * index_scale * sum_d |q_d k_d| (twice that bound).
Which columns are scored, -inf or left unwritten must match exactly.
"""

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu


def _bf16(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_gpu(iw, st, init, local, scale, score_cols, iq=None, cache=None, flags=0):
    import torch

    from indexer_projection_gb300 import binding as B

    dev = torch.device("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    d_iq = t(st["iq"].view(np.int16)) if iq is None else iq
    d_cache = t(st["index_cache"]) if cache is None else cache
    d_bt, d_sl = t(st["block_table"]), t(st["seq_lens"])
    scores = torch.full((iw.M, score_cols), float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    a = B.pa_index_args(B.ptr(d_iq), d_iq.shape[1], iw.head, B.ptr(d_cache), d_cache.numel() // 128,
                        B.ptr(d_bt), B.ptr(d_sl), iw.R, iw.q_len, st["block_table"].shape[1], init, local,
                        scale, B.ptr(scores), score_cols, B.ptr(status), flags)
    B.pre_attn_index_scores(a, torch.cuda.current_stream())
    torch.cuda.synchronize()
    return scores.cpu().numpy(), int(status.item())


def compare_scores(iw, st, got, want, scale, iq_bits=None, extra_abs=None):
    assert got.shape == want.shape
    assert np.array_equal(np.isnan(got), np.isnan(want)), "written columns differ"
    assert np.array_equal(np.isneginf(got), np.isneginf(want)), "-inf columns differ"
    lut = np.array([oracle.e4m3_decode(c) for c in range(256)], np.float64)
    lut[np.isnan(lut)] = 0
    keys = np.abs(lut[st["index_cache"].reshape(-1, 128)])
    iq = st["iq"] if iq_bits is None else iq_bits
    q = np.abs(_bf16(iq[:, iw.head * 128:(iw.head + 1) * 128]))
    n = 0
    for r in range(iw.R):
        rows = slice(r * iw.q_len, (r + 1) * iw.q_len)
        fin = np.isfinite(want[rows])
        cols = np.nonzero(fin.any(axis=0))[0]
        if cols.size == 0:
            continue
        slots = st["block_table"][r, cols // 128].astype(np.int64) * 128 + cols % 128
        l1 = q[rows] @ keys[slots].T  # sum_d |q_d k_d| for each (row, key)
        tol = 2.0 ** -16 * abs(scale) * l1 + 1e-30
        if extra_abs is not None:
            tol = tol + extra_abs[rows] @ keys[slots].T * abs(scale)
        g, w = got[rows][:, cols], want[rows][:, cols]
        m = fin[:, cols]
        err = np.abs(g.astype(np.float64)[m] - w[m]) - tol[m]
        assert np.all(err <= 0), f"request {r}: max excess {err.max():.3g}"
        n += int(m.sum())
    return n


def check(iw, init=1, local=4, score_cols=None):
    st = workloads.index_host_state(iw)
    scale = float(np.float32(oracle.index_scale_log2e(iw.sm_scale)))
    cols = st["block_table"].shape[1] * 128 if score_cols is None else score_cols
    got, status = run_gpu(iw, st, init, local, scale, cols)
    assert status == 0
    iq = st["iq"]
    want = oracle.index_scores(iq[:, iw.head * 128:(iw.head + 1) * 128], st["index_cache"], st["block_table"],
                               st["seq_lens"], iw.q_len, init, local, scale, cols)
    n = compare_scores(iw, st, got, want, scale)
    assert n > 0
    return n


def test_decode_config():
    check(workloads.index_decode())


def test_spec_decode_config():
    check(workloads.index_spec_decode())


@pytest.mark.parametrize("q_len,init,local", [(1, 0, 0), (7, 1, 4), (13, 2, 3), (16, 0, 1), (9, 3, 0)])
def test_row_counts_and_pinned_blocks(q_len, init, local):
    iw = workloads.IndexWorkload(f"ix{q_len}", R=5, q_len=q_len, seq_lo=q_len, seq_hi=2000, bt_width=20,
                                 seed=q_len + 10 * init + local, n_iq=2, head=1)
    check(iw, init, local, score_cols=20 * 128 + 64)


def test_short_requests_and_wide_rows():
    # seq_len == q_len (the first rows of a request), single partial blocks,
    # and score rows wider than the block table
    iw = workloads.IndexWorkload("ixs", R=6, q_len=3, seq_lo=3, seq_hi=400, bt_width=4, seed=5)
    check(iw, 0, 1, score_cols=1024)


def test_block_ids_outside_the_cache_are_skipped_and_flagged():
    from indexer_projection_gb300 import binding as B

    iw = workloads.IndexWorkload("ixbad", R=3, q_len=2, seq_lo=600, seq_hi=900, bt_width=8, seed=9)
    st = workloads.index_host_state(iw)
    nslots = st["index_cache"].size // 128
    st["block_table"][1, 2] = nslots // 128 + 7  # beyond the cache
    scale = 0.125
    got, status = run_gpu(iw, st, 0, 0, scale, 8 * 128)
    assert status == B.PA_DEV_SLOT_RANGE
    assert np.all(np.isnan(got[2:4, 256:384]))    # request 1's bad block: not written
    good = [0, 1, 4, 5]
    want = oracle.index_scores(st["iq"][good], st["index_cache"], st["block_table"][[0, 2]], st["seq_lens"][[0, 2]],
                               iw.q_len, 0, 0, scale, 8 * 128)
    iw2 = workloads.IndexWorkload("ixgood", R=2, q_len=2, seq_lo=1, seq_hi=2, bt_width=8, seed=0)
    st2 = {"iq": st["iq"][good], "index_cache": st["index_cache"], "block_table": st["block_table"][[0, 2]]}
    compare_scores(iw2, st2, got[good], want, scale)


def test_scores_follow_the_step_on_the_same_stream():
    # pre_attn_run writes the step's index_q and new index keys, then the
    # scorer runs behind it on the same stream; the oracle does the same
    # from the same inputs.  The scores then differ only by what the two
    # index_q rows may differ by (bf16 within 1e-2 + 2e-2 |q|), which the
    # tolerance adds, and by the keys' one-code steps, which this check
    # leaves out by comparing the keys the oracle wrote
    import torch

    from tests import harness

    R, bt_width = 8, 64
    g = np.random.default_rng(3)
    wl = workloads.decode().replace(pool_pages16=R * bt_width * 8 + 64)
    st = workloads.host_state(wl)
    seq = g.integers(1, bt_width * 128, R).astype(np.int32)
    bt = g.permutation(R * bt_width).reshape(R, bt_width).astype(np.int32)
    pos = (seq - 1).astype(np.int64)
    st["positions"] = pos
    st["slot_mapping"] = (bt[np.arange(R), pos // 128].astype(np.int64) * 128 + pos % 128)
    st["index_slot_mapping"] = st["slot_mapping"].copy()
    keys = workloads._e4m3_bits(torch.randn(wl.num_index_slots, 128, generator=torch.Generator().manual_seed(4)))
    st["index_cache"] = keys.reshape(-1)
    gr = harness.GpuRun(wl, st)
    gr.run()
    iw = workloads.IndexWorkload("ixstep", R=R, q_len=1, seq_lo=1, seq_hi=2, bt_width=bt_width, seed=0)
    scale = float(np.float32(oracle.index_scale_log2e(iw.sm_scale)))
    ist = {"block_table": bt, "seq_lens": seq}
    got, status = run_gpu(iw, ist, 1, 4, scale, bt_width * 128, iq=gr.d["iq_bf16"], cache=gr.d["index_cache"])
    assert status == 0
    ref = harness.oracle_run(wl, st, range(wl.M))
    want = oracle.index_scores(ref["iq_bf16"], ref["index_cache"], bt, seq, 1, 1, 4, scale, bt_width * 128)
    gpu_cache = gr.results()["index_cache"]
    # the new keys may sit one code apart; score the oracle's rows against
    # the GPU's cache only where the two caches agree
    same = np.array_equal(gpu_cache, ref["index_cache"])
    cmp = {"iq": ref["iq_bf16"], "index_cache": ref["index_cache"], "block_table": bt}
    dq = 1e-2 + 2e-2 * np.abs(_bf16(ref["iq_bf16"]))
    if same:
        compare_scores(iw, cmp, got, want, scale, extra_abs=dq)
    else:
        assert np.array_equal(np.isnan(got), np.isnan(want)) and np.array_equal(np.isneginf(got), np.isneginf(want))


def test_many_requests_take_the_per_request_grid():
    # more than 512 requests: the per-request grid, not the persistent kernel
    iw = workloads.IndexWorkload("ixmany", R=600, q_len=2, seq_lo=2, seq_hi=700, bt_width=6, seed=17)
    check(iw, 1, 1)


def test_persistent_slices_cross_requests_and_empty_ones():
    # requests of one row and very different lengths (some whose only block is
    # pinned), so CTA slices start and end inside requests and skip empty ones
    iw = workloads.IndexWorkload("ixmix", R=300, q_len=1, seq_lo=1, seq_hi=6000, bt_width=47, seed=19)
    check(iw, 1, 2)


@pytest.mark.parametrize("R", [5, 600])
def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_correct(R):
    # PA_FLAG_TEST_WAIT_TIMEOUT: the score warps also wait on a barrier
    # nothing arrives on (200 us limit); every CTA stops, no scored key is
    # written, PA_DEV_WAIT_TIMEOUT comes back, and a normal call after it (the
    # persistent kernel at R = 5, the per-request grid at R = 600) is exact
    from indexer_projection_gb300 import binding as B

    iw = workloads.IndexWorkload(f"ixto{R}", R=R, q_len=2, seq_lo=200, seq_hi=1500, bt_width=12, seed=70 + R)
    st = workloads.index_host_state(iw)
    scale = float(np.float32(oracle.index_scale_log2e(iw.sm_scale)))
    cols = st["block_table"].shape[1] * 128
    got, status = run_gpu(iw, st, 1, 1, scale, cols, flags=B.PA_FLAG_TEST_WAIT_TIMEOUT)
    assert status & B.PA_DEV_WAIT_TIMEOUT
    want = oracle.index_scores(st["iq"][:, iw.head * 128:(iw.head + 1) * 128], st["index_cache"],
                               st["block_table"], st["seq_lens"], iw.q_len, 1, 1, scale, cols)
    scored = np.isfinite(want)
    assert not np.any(np.isfinite(got) & scored)  # no scored key was written
    check(iw, 1, 1)


@pytest.mark.parametrize("R", [5, 600])
def test_query_values_off_the_f16_grid_take_the_bf16_path(R):
    # a warp's fragments go to f16 MMAs only when every query value is an
    # f16 value (0, or 2^-17 <= |x| < 2^15); here request 1 has one value of
    # 40000 and request 3 one of 1e-7 (their warps keep the bf16 path), the
    # others stay on the f16 path: all scores follow the oracle
    iw = workloads.IndexWorkload(f"ixgrid{R}", R=R, q_len=3, seq_lo=300, seq_hi=2000, bt_width=16, seed=77)
    st = workloads.index_host_state(iw)
    iq = st["iq"].copy()  # bf16 bits
    big = np.array([40000.0], np.float32).view(np.uint32) >> 16
    tiny = np.array([1e-7], np.float32).view(np.uint32) >> 16
    iq[1 * iw.q_len + 1, iw.head * 128 + 5] = np.uint16(big[0])
    iq[3 * iw.q_len + 0, iw.head * 128 + 77] = np.uint16(tiny[0])
    st["iq"] = iq
    scale = float(np.float32(oracle.index_scale_log2e(iw.sm_scale)))
    cols = st["block_table"].shape[1] * 128
    got, status = run_gpu(iw, st, 1, 2, scale, cols)
    assert status == 0
    want = oracle.index_scores(iq[:, iw.head * 128:(iw.head + 1) * 128], st["index_cache"], st["block_table"],
                               st["seq_lens"], iw.q_len, 1, 2, scale, cols)
    assert compare_scores(iw, st, got, want, scale, iq_bits=iq) > 0
