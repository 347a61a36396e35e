"""The multi-GPU mode is replicas only (batch-1 decoding of one request does not shard without a
per-layer all-reduce): each rank runs its own request, the job's time is the slowest rank's and the
throughput counts every rank's tokens.  The host side of that is checked here with world_size-2
gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 150.0][rank]
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        out[rank] = (ms, bench.job_throughput(255 * 3, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_count_all_tokens():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        got = dict(out)
    assert got[0] == got[1]
    ms, value = got[0]
    assert ms == 150.0
    assert value == pytest.approx(255 * 3 * 2 / 0.150)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(42.0, 1) == 42.0
    assert bench.job_throughput(100, 1, 500.0) == pytest.approx(200.0)
