"""The benchmark's several-rank path on CPU: two gloo ranks agree on the
slowest rank's times and the whole-job throughput (the GPU path does the same
over NCCL, one process per GPU, each an independent replica of the step)."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (r + 1) ms a step and an e2e time of 10 - r ms
        got = bench.max_over_ranks([rank + 1.0, 10.0 - rank], world)
        q.put((rank, got, bench.tokens_per_second(world, 8, got[0])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, tps in res:
        assert got == [2.0, 10.0]
        assert tps == pytest.approx(2 * 8 / 2e-3)


def test_one_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks([3.5], 1) == [3.5]
    assert bench.tokens_per_second(1, 8, 8e-3) == pytest.approx(1e6)
