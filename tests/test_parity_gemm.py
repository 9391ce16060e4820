"""GPU parity of the tensor-core path (prologue + persistent tcgen05 GEMM with
the fused head epilogue) against the CPU oracle, through the C-ABI.  Small
cases compare every row; the full-size configurations compare sampled rows
(tile boundaries, first and last rows, random rows) and check that no byte
outside the written slots changed."""

import numpy as np
import pytest

import workloads
from tests import harness

pytestmark = pytest.mark.gpu


def _flags(force_gemm=True):
    from indexer_projection_gb300 import binding as B
    return B.PA_FLAG_FORCE_GEMM if force_gemm else 0


def check(wl, rows=None, flags=None, gemm_grid=0, nsample=48):
    st = workloads.host_state(wl)
    g = harness.GpuRun(wl, st, flags=_flags() if flags is None else flags, gemm_grid=gemm_grid)
    g.run()
    got = g.results()
    if rows is None:
        rows = list(range(wl.M)) if wl.M <= 512 else harness.sample_rows(wl.M, nsample, seed=wl.seed)
    ref = harness.oracle_run(wl, st, rows)
    tally = harness.compare(wl, got, ref, rows, all_rows=range(wl.M))
    assert g.runner.device_status() == 0
    return tally


def small(name, M, fmt="ptpc", cache="fp8", nkv=1, H=512, seed=21, **kw):
    base = dict(positions="uniform", max_pos=4096, pool_pages16=2048, pool_pages=512, q_fp8=True, iq_fp8=True)
    base.update(kw)
    return workloads.Workload(name, H=H, nkv=nkv, M=M, weight_fmt=fmt, cache_fmt=cache, seed=seed, **base)


@pytest.mark.parametrize("fmt", ["ptpc", "mx"])
@pytest.mark.parametrize("cache", ["fp8", "nvfp4"])
def test_small_ragged(fmt, cache):
    check(small(f"g_{fmt}_{cache}", 200, fmt, cache, nkv=2, skip_rows=(3, 130)))


@pytest.mark.parametrize("M", [1, 5, 17, 127, 128, 129, 256])
def test_token_counts(M):
    check(small(f"g_m{M}", M, "mx", "nvfp4", H=1024, seed=M))


@pytest.mark.parametrize("grid", [1, 3, 37])
def test_persistent_grid_override(grid):
    # fewer CTAs than tiles: every CTA walks many tiles through both TMEM buffers
    check(small(f"g_grid{grid}", 300, "mx", "fp8", nkv=1, H=768, seed=grid), gemm_grid=grid)


def test_long_k_and_outliers():
    check(small("g_k6144", 136, "ptpc", "fp8", nkv=1, H=6144, seed=8, outlier_frac=0.05))


def test_spec_decode_config():
    check(workloads.spec_decode(), flags=0)


def test_prefill_config():
    check(workloads.prefill(), flags=0, nsample=40)


@pytest.mark.parametrize("M", [64, 256, 1024, 4096, 16384])
def test_sweep_config_tensor_core_points(M):
    check(workloads.sweep(M), flags=0, nsample=24)
