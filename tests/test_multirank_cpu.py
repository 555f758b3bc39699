"""The bench's multi-rank aggregation with two gloo ranks on the CPU: the
timed region's duration is the max over ranks and the throughput counts every
rank's tokens over that time."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 100.0 + 50.0 * rank  # rank 1 is the slow one
        m = bench.reduce_max(ms)
        out[rank] = (m, bench.whole_job_tokens_per_s(1000, world, m), bench.dist_setup())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        m, v, (world, rank, _) = out[r]
        assert m == 150.0
        assert v == pytest.approx(2 * 1000 / 0.150)
        assert (world, rank) == (2, r)


def test_single_process_needs_no_group():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.whole_job_tokens_per_s(65536, 1, 100.0) == pytest.approx(655360.0)
