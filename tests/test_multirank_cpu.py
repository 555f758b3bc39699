"""The bench's multi-rank aggregation with two gloo ranks on the CPU: the
timed region's duration is the max over ranks, the throughput counts every
rank's tokens over that time, and the decision to measure again after a
rejected clock record is taken by all ranks together.  The bench's own rank
launcher (``--gpus N`` outside torchrun) starts the ranks; run as a script
under it, this file is one gloo rank that prints the whole-job line."""

import json
import os
import socket
import subprocess
import sys

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


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _json_lines(text):
    out = []
    for ln in text.splitlines():
        ln = ln.strip()
        if ln.startswith("{"):
            out.append(json.loads(ln))
    return out


def test_launcher_starts_two_gloo_ranks():
    """bench.launch_ranks (what ``--gpus N`` uses) starts two ranks of a script; they
    aggregate over gloo and rank 0 alone prints one line with n_gpus = 2."""
    code = ("import sys; sys.path.insert(0, %r); import bench; "
            "sys.exit(bench.launch_ranks(2, [%r]))" % (ROOT, os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["n_gpus"] == 2 and line["ranks_seen"] == [0, 1]
    assert line["ms_per_step"] == 150.0 and line["value"] == pytest.approx(2 * 1000 / 0.150)


def test_bench_gpus_flag_spawns_ranks_for_the_reference_arm():
    """``bench.py --impl reference --gpus 2`` outside torchrun goes through the same
    launcher: two ranks start, rank 0 alone times the oracle and prints one line."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "tiny", "--steps", "1", "--warmup", "3", "--ref-step-seconds", "0.2"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1, r.stdout
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2
    assert lines[0]["ms_per_step"] < 60_000.0  # the measured wall time of one bounded step


def test_bench_gpus_flag_without_enough_gpus_fails():
    """``--gpus 2`` where fewer than two GPUs are visible exits non-zero and prints no
    line (never an N = 1 line under an N = 2 request)."""
    import torch
    if torch.cuda.device_count() >= 2:
        pytest.skip("two GPUs are visible here")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode != 0
    assert not _json_lines(r.stdout)
    assert "needs 2 visible GPUs" in r.stderr


def _rank_main():
    """One rank under bench.launch_ranks: gloo process group from the launcher's
    environment, the bench's max-over-ranks and whole-job throughput, one line from rank 0."""
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench
    world, rank, _ = bench.dist_setup()
    dist.init_process_group("gloo")
    ms = 100.0 + 50.0 * rank
    m = bench.reduce_max(ms)
    ranks = [None] * world
    dist.all_gather_object(ranks, rank)
    if rank == 0:
        print(json.dumps({"n_gpus": world, "ms_per_step": m, "ranks_seen": sorted(ranks),
                          "value": bench.whole_job_tokens_per_s(1000, world, m)}), flush=True)
    dist.barrier()
    dist.destroy_process_group()
    del torch


if __name__ == "__main__":
    _rank_main()
