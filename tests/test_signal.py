"""Signal mode and bounded device waits, on the GPU, through the C-ABI.

Signal mode (the pre_attn page's done flags, emit_pre_attn.publish_done):
every (token, head) row of the step sets its done word to the step's epoch
once its outputs and cache bytes are written, with release semantics; the
library's consumer kernel (pre_attn_wait_done) waits for the words with
acquire loads and a bounded limit.

Failure detection without a GPU fault: a wait that nothing can satisfy runs
out after a short limit, the kernel raises PA_DEV_WAIT_TIMEOUT in a status
word the host reads and returns; the context stays usable and the next step
is correct.
"""

import numpy as np
import pytest

import workloads
from tests import harness

pytestmark = pytest.mark.gpu


def _flags(path):
    from indexer_projection_gb300 import binding as B
    return {"skinny": B.PA_FLAG_FORCE_GEMV, "persist": B.PA_FLAG_FORCE_GEMV | B.PA_FLAG_GEMV_PERSIST,
            "single": B.PA_FLAG_FORCE_GEMM | B.PA_FLAG_GEMM_SINGLE,
            "pair": B.PA_FLAG_FORCE_GEMM | B.PA_FLAG_GEMM_PAIR}[path]


def _wl(path):
    if path in ("skinny", "persist"):
        return workloads.tiny().replace(M=5, q_fp8=True, iq_fp8=True, skip_rows=(2,))
    return workloads.tiny().replace(name=f"sig_{path}", M=100, weight_fmt="mx", cache_fmt="nvfp4", pool_pages=64,
                                    q_fp8=True, iq_fp8=True, skip_rows=(7,))


@pytest.mark.parametrize("path", ["skinny", "persist", "single", "pair"])
def test_done_words_carry_the_epoch_of_each_step(path):
    wl = _wl(path)
    st = workloads.host_state(wl)
    g = harness.GpuRun(wl, st, flags=_flags(path))
    for epoch in (7, 8):
        g.set_done_epoch(epoch)
        g.run()
        got = g.results()
        words = g.done.cpu().numpy().view(np.uint32)
        assert words.shape == (wl.M * wl.n_heads,)
        assert np.all(words == epoch), np.unique(words)  # every row, skipped cache slots included
        ref = harness.oracle_run(wl, st, range(wl.M))
        harness.compare(wl, got, ref, range(wl.M))
        assert g.runner.device_status() == 0


@pytest.mark.parametrize("path", ["skinny", "persist", "pair"])
def test_consumer_chained_behind_the_step_sees_every_word(path):
    from indexer_projection_gb300 import binding as B

    wl = _wl(path)
    st = workloads.host_state(wl)
    g = harness.GpuRun(wl, st, flags=_flags(path))
    status = g.torch.zeros(1, dtype=g.torch.int32, device=g.dev)
    stream = g.torch.cuda.current_stream()
    for epoch in (11, 12, 13):
        g.set_done_epoch(epoch)
        g.run()
        # launched with programmatic dependent launch right behind the step: it
        # may start while the step's last kernel runs and follows the words
        B.pre_attn_wait_done(g.done, wl.M * wl.n_heads, epoch, 1_000_000, status, stream)
    g.torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.all(g.done.cpu().numpy().view(np.uint32) == 13)


def test_consumer_wait_runs_out_and_the_stream_stays_usable():
    from indexer_projection_gb300 import binding as B

    wl = _wl("skinny")
    st = workloads.host_state(wl)
    g = harness.GpuRun(wl, st, flags=_flags("skinny"))
    status = g.torch.zeros(1, dtype=g.torch.int32, device=g.dev)
    never = g.torch.zeros(300, dtype=g.torch.int32, device=g.dev)  # nothing writes these words
    B.pre_attn_wait_done(never, 300, 5, 100, status, g.torch.cuda.current_stream())
    g.torch.cuda.synchronize()
    assert int(status.item()) == B.PA_DEV_WAIT_TIMEOUT
    g.run()
    ref = harness.oracle_run(wl, st, range(wl.M))
    harness.compare(wl, g.results(), ref, range(wl.M))
    # argument errors are refused before anything is launched
    assert B.pre_attn_wait_done(never, 0, 5, 100, status, check=False) == B.PA_ERR_SHAPE
    assert B.pre_attn_wait_done(never, 3, 0, 100, status, check=False) == B.PA_ERR_CONFIG
    assert B.pre_attn_wait_done(never, 3, 5, 0, status, check=False) == B.PA_ERR_CONFIG
    assert B.pre_attn_wait_done(None, 3, 5, 100, status, check=False) == B.PA_ERR_NULL


@pytest.mark.parametrize("path", ["skinny", "persist", "single", "pair"])
def test_a_device_wait_that_runs_out_is_reported_and_the_next_step_is_correct(path):
    # PA_FLAG_TEST_WAIT_TIMEOUT: the main kernel's epilogue waits on a barrier
    # nothing arrives on, with a 200 us limit; the wait runs out, the kernel
    # skips the rows' stores and done words, raises PA_DEV_WAIT_TIMEOUT and
    # returns (freeing its tensor memory)
    from indexer_projection_gb300 import binding as B

    wl = _wl(path)
    st = workloads.host_state(wl)
    g = harness.GpuRun(wl, st, flags=_flags(path) | B.PA_FLAG_TEST_WAIT_TIMEOUT)
    g.set_done_epoch(3)
    g.run()
    got = g.results()
    assert g.runner.device_status() & B.PA_DEV_WAIT_TIMEOUT
    assert np.all(g.done.cpu().numpy() == 0)                # no row was published
    assert np.all(got["q_bf16"] == 0xA5A5)                   # nor written
    # the same context, a handle without the testing flag: a correct step
    g2 = harness.GpuRun(wl, st, flags=_flags(path))
    g2.run()
    ref = harness.oracle_run(wl, st, range(wl.M))
    harness.compare(wl, g2.results(), ref, range(wl.M))
    assert g2.runner.device_status() == 0
