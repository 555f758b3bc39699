"""The bench's multi-rank aggregation with two gloo ranks on the CPU: the
timed region's duration is the max over ranks, the throughput counts every
rank's tokens over that time, and the decision to measure again after a
rejected clock record is taken by all ranks together."""

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
        # only rank 1's GPU saw a thermal slowdown; both ranks must measure again
        clk = {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0,
               "reasons": ["sw_power_cap"] + (["hw_thermal_slowdown"] if rank == 1 else [])}
        again = bench.reduce_max(1.0 if bench.clocks_rejected(clk) else 0.0) > 0.0
        out[rank] = (m, bench.whole_job_tokens_per_s(1000, world, m), bench.dist_setup(), again)
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
        m, v, (world, rank, _), again = out[r]
        assert m == 150.0
        assert v == pytest.approx(2 * 1000 / 0.150)
        assert (world, rank) == (2, r)
        assert again


def test_single_process_needs_no_group():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.whole_job_tokens_per_s(65536, 1, 100.0) == pytest.approx(655360.0)


def test_clock_records_the_timing_rules_reject():
    import bench
    ok = {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert not bench.clocks_rejected(ok)                      # a power cap is kept and noted
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected(dict(ok, reasons=["sw_power_cap", r]))
    assert bench.clocks_rejected({"sm_mhz": 900.0, "sm_max_mhz": 2070.0, "reasons": []})   # a leftover lock
    assert not bench.clocks_rejected({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []})
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0})


def test_rows_the_backward_contracts():
    import numpy as np

    import bench
    from workloads import generate, workload
    inp = generate("rlpg", T=1000, Hd=64, V=500, n_seq=4)
    valid = inp.targets != inp.ignore_index
    assert bench.kept_rows(inp, workload("rlpg")) == int(np.count_nonzero(valid & (inp.dloss != 0)))
    inp2 = generate("medium", T=1000, Hd=64, V=500)
    assert bench.kept_rows(inp2, workload("medium")) == int(np.count_nonzero(inp2.targets != inp2.ignore_index))
