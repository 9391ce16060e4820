"""pre_attn_run_noalloc, the entry point for callers that cannot allocate
device memory (a plugin whose host runtime owns every byte of device memory,
a process whose device memory is capped after start-up), against
pre_attn_run with a caller workspace.

Kept in a file pytest collects last, so that a run stopping at its first
failure has run every other test before this one.  It passes on its own in a
fresh process and after the rest of the suite: the entry point clears the
part of its shared static scratch that must start at zero on every call.
"""

import numpy as np
import pytest

import workloads
from tests import harness

pytestmark = pytest.mark.gpu


def _inputs(B, d):
    return B.pa_step_inputs(B.ptr(d["ar"]), B.ptr(d["res"]), B.ptr(d["positions"]), B.ptr(d["slot_mapping"]),
                            B.ptr(d["index_slot_mapping"]))


def _expected_and_noalloc(wl, st=None):
    from indexer_projection_gb300 import binding as B

    st = workloads.host_state(wl) if st is None else st
    ref = harness.GpuRun(wl, st)  # the existing entry point, caller workspace
    ref.run()
    want = ref.results()
    g = harness.GpuRun(wl, st)    # fresh copies of the same inputs, caches and outputs
    stream = g.torch.cuda.current_stream()
    assert B.pre_attn_run_noalloc(g.runner.handle, wl.M, _inputs(B, g.d), g.weights, g.caches, g.outputs,
                                  stream) == B.PA_OK
    got = g.results()
    return st, want, got, B.pre_attn_noalloc_status(stream)


def test_noalloc_matches_pre_attn_run_on_two_calls_in_a_row():
    # two calls back to back on different shapes: the second finds the first
    # one's contents in the shared scratch.  Both entry points run the same
    # kernels on the same inputs, so every output and cache byte is equal.
    for wl in (workloads.decode().replace(q_fp8=True, iq_fp8=True),
               workloads.tiny().replace(M=13, nkv=2, n_q=0, n_iq=0, weight_fmt="mx", seed=17, iq_fp8=True)):
        st, want, got, status = _expected_and_noalloc(wl)
        assert status == 0
        assert set(want) == set(got)
        for k in want:
            assert np.array_equal(want[k].view(np.uint8), got[k].view(np.uint8)), k


def test_noalloc_status_reports_the_last_call():
    from indexer_projection_gb300 import binding as B

    wl = workloads.tiny().replace(M=4)
    st = workloads.host_state(wl)
    st["slot_mapping"][1] = wl.num_pages16 * 16 + 5   # beyond the cache: the store is skipped and flagged
    _, want, got, status = _expected_and_noalloc(wl, st)
    assert status == B.PA_DEV_SLOT_RANGE
    for k in want:
        assert np.array_equal(want[k].view(np.uint8), got[k].view(np.uint8)), k
    # the next call starts from a cleared status word
    _, _, _, status = _expected_and_noalloc(workloads.tiny().replace(M=3, seed=5))
    assert status == 0


def test_noalloc_rejects_rows_it_cannot_take():
    from indexer_projection_gb300 import binding as B
    from indexer_projection_gb300.runner import PreAttn

    wl = workloads.tiny()
    st = workloads.host_state(wl)
    g = harness.GpuRun(wl, st, max_tokens=32)
    d = g.d
    ins = B.pa_step_inputs(B.ptr(d["ar"]), B.ptr(d["res"]), B.ptr(d["positions"]), B.ptr(d["slot_mapping"]), None)
    # M beyond 16 rows
    assert B.pre_attn_run_noalloc(g.runner.handle, 17, ins, g.weights, g.caches, g.outputs, check=False) \
        == B.PA_ERR_SHAPE
    # beyond the handle's max_tokens
    small = PreAttn(512, 1, weight_format=B.PA_WEIGHT_FP8_PER_CHANNEL, cache_format=B.PA_CACHE_FP8, max_tokens=4)
    assert B.pre_attn_run_noalloc(small.handle, 5, ins, g.weights, g.caches, g.outputs, check=False) \
        == B.PA_ERR_SHAPE
    # the largest request the handles accept (H = 16384, MXFP8, 16 rows)
    # needs well under the 2 MiB: the scratch holds only the activations
    big = PreAttn(16384, 4, weight_format=B.PA_WEIGHT_MXFP8, cache_format=B.PA_CACHE_FP8,
                  max_tokens=16, n_q_heads=250, n_iq_heads=5)
    assert 0 < B.pre_attn_workspace_bytes(big.handle, 16) <= (2 << 20)
