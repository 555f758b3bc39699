#!/usr/bin/env python3
"""Benchmark: fused linear cross-entropy forward + backward on GB300.

One step = flce_forward + flce_backward over one batch of the workload (all
steps of the path: logit tiles with the log-sum-exp epilogue, finalize, dZ
recompute, dH and dW contractions).  The default workload is 65,536 tokens x
hidden 2048 x vocab 124,160 (bf16 inputs, fp32 accumulation).

Prints one JSON line.  ``value`` is whole-job tokens/s with the inputs resident
in HBM; ``e2e`` is the same metric through the public API with the inputs in
pinned host memory, copied in, and the loss and per-token log p(target) copied
back, inside the timed region (dH and dW stay on the device for the optimizer).
``--impl reference`` times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload).

Multi-GPU (torchrun): every rank runs its own replica of the workload (the op
shards by token batches with no exchange inside it), the timed region is
bracketed by barriers, and the max over ranks is reported.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import generate, workload  # noqa: E402

METRIC = "fused linear-CE fwd+bwd tokens/s (T=64K,V=124,160); % of GB300 BF16 TC peak"
DEFAULT_WORKLOAD = "lmhead_T65536_H2048_V124160"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return json.load(fh), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha():
    """Hash of the library's code with comments and whitespace removed, so that
    DRAM counters stay attached to the code they were taken on."""
    import re
    h = hashlib.sha256()
    for f in ("csrc/flce_kernels.cuh", "csrc/ptx.cuh", "csrc/flce_api.cu"):
        with open(os.path.join(ROOT, "lm_head_linear_gb300", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel, T, Hd, V, chunk=None, launches_per_step=1):
    """DRAM bytes per launch of `kernel` at T x Hd x V, from the committed ncu summary of
    a smaller case (profiles/traffic.json), if it was taken on the current kernel sources
    (else None).  The backward kernels work on one token chunk per launch; at the same
    chunk and Hd their traffic grows in proportion to V, so the small case's medians are
    scaled by V / V_case, the first chunk's (dW stored) and the later chunks' (dW
    reduce-added) weighted by the run's launches per step.  The forward's traffic does not
    grow in proportion to its tiles (it depends on which operand blocks stay in L2), so it
    is reported only for the captured shape itself."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        data = json.load(fh)
    if data.get("source_sha") != kernel_source_sha():
        return None
    case = data.get("case", {})
    rec = data.get("kernels", {}).get(kernel)
    if not rec or case.get("Hd") != Hd:
        return None
    if rec.get("scale") == "V":
        if chunk != case.get("chunk"):
            return None
        n = max(int(launches_per_step), 1)
        first, later = float(rec["first_chunk"]["median"]), float(rec["later_chunks"]["median"])
        return (first + (n - 1) * later) / n * V / float(case["V"])
    return float(rec["median"]) if (case.get("T"), case.get("V")) == (T, V) else None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def clocks_rejected(c):
    """True for a clock record the timing rules reject: hardware or thermal slowdown, or
    a median SM clock far below the maximum with no throttle reason active."""
    if set(c.get("reasons", [])) & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}:
        return True
    sm, mx = c.get("sm_mhz"), c.get("sm_max_mhz")
    return bool(sm and mx and not c.get("reasons") and sm < 0.7 * mx)


def reduce_max(x, device=None):
    """Max of a float over the ranks of the default process group (x itself when
    there is none).  NCCL reduces a tensor on `device`, gloo one on the CPU."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    on = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_rank, world, max_ms):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (max_ms / 1000.0)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def free_port():
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_ranks(nprocs, argv, env=None):
    """Runs ``argv`` (a script and its arguments) as ``nprocs`` ranks of one node through
    torch.distributed.run, with the rendezvous on 127.0.0.1; every rank gets RANK,
    LOCAL_RANK and WORLD_SIZE.  Returns the launcher's exit code (non-zero when a rank
    failed)."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={int(nprocs)}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", *argv]
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.call(cmd, env=e)


def spawn_self(args):
    """``--gpus N`` (N > 1) outside a launcher: start N ranks of this script, one per GPU.
    The replicas exchange nothing on the data path; NCCL carries the barriers and the
    max-over-ranks reduction of the timed region, and its communicator lines are printed
    (NCCL_DEBUG=INFO for the INIT subsystem unless the caller set NCCL_DEBUG)."""
    if args.impl == "ours":
        import torch
        have = torch.cuda.device_count()
        if have < args.gpus:
            print(f"bench.py: --gpus {args.gpus} needs {args.gpus} visible GPUs, this process sees {have}",
                  file=sys.stderr, flush=True)
            return 2
    env = {}
    if "NCCL_DEBUG" not in os.environ:
        env = {"NCCL_DEBUG": "INFO", "NCCL_DEBUG_SUBSYS": "INIT"}
    return launch_ranks(args.gpus, [os.path.abspath(__file__), *sys.argv[1:]], env)


def time_oracle(inp, budget_s=12.0, slice_tokens=128, W64=None):
    """Tokens/s of the fp64 oracle (as it stands) on slices of the workload's tokens:
    forward + backward for each slice with the full vocabulary."""
    import oracle
    if W64 is None:
        W64 = inp.W64()
    t_start = time.perf_counter()
    done = 0
    s0 = 0
    while True:
        rows = np.arange(s0, min(s0 + slice_tokens, inp.T))
        H64 = inp.H64(rows)
        y = inp.targets[rows]
        dl = inp.dloss[rows] if inp.reduction == "none" else inp.dloss
        oracle.forward(H64, W64, y, inp.ignore_index, inp.reduction)
        oracle.backward(dl, H64, W64, y, inp.ignore_index, inp.reduction)
        done += len(rows)
        s0 = (s0 + slice_tokens) % inp.T
        el = time.perf_counter() - t_start
        if el >= budget_s:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": done / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} tokens in {slice_tokens}-token slices, forward + backward over the full "
                      f"V={inp.V}, Hd={inp.Hd}, fp64 numpy, {el:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    wl = workload(args.workload)
    inp = generate(wl, T=args.T, Hd=args.Hd, V=args.V)
    W64 = inp.W64()
    for _ in range(args.warmup):
        time_oracle(inp, budget_s=0.0, slice_tokens=32, W64=W64)
    per = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        per.append(time_oracle(inp, budget_s=args.ref_step_seconds, slice_tokens=64, W64=W64))
    el = time.perf_counter() - t0
    value = sum(r["value"] for r in per) / len(per)
    tokens = value * el
    # Each timed step is a bounded sample (a few seconds of token slices), so ms_per_step is
    # the measured wall time of one such step; the time the oracle would take for the whole
    # batch of T tokens at the same rate is reported beside it.
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * el / args.steps,
        "ms_per_full_batch_extrapolated": 1000.0 * inp.T / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "T": inp.T, "Hd": inp.Hd, "V": inp.V,
                                        "reduction": wl.reduction},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": per[0]["cores"], "kind": "oracle",
                         "sample": f"each step: {per[0]['sample']}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "tokens_timed": int(tokens),
    }
    print(json.dumps(line), flush=True)
    return 0


class LossPath:
    """The hot path: flce_forward + flce_backward (8·T·Hd·V FLOPs per step).  Inputs H, W,
    targets, dloss; the loss and per-token logp are read back, dH and dW stay on the device."""

    name = "loss"

    def __init__(self, flce, torch, inp, wl, dev, args):
        self.flce, self.torch, self.inp, self.wl, self.dev = flce, torch, inp, wl, dev
        T, Hd, V = inp.T, inp.Hd, inp.V
        self.metric = METRIC
        self.flops_per_step = 8.0 * T * Hd * V
        self.flops_executed_per_step = (2.0 * T + 6.0 * kept_rows(inp, wl)) * Hd * V
        self.host = host_inputs(torch, inp, with_dloss=True)
        self.ins = tuple(t.to(dev) for t in self.host)
        self.fws = torch.empty(flce.flce_forward_workspace_size(T, Hd, V), dtype=torch.uint8, device=dev)
        bws_bytes = flce.flce_backward_workspace_size(T, Hd, V)
        if args.bwd_chunk:
            # a workspace for chunks of `bwd_chunk` rows (the library sizes its chunk from
            # the workspace it is given)
            bws_bytes = flce.flce_backward_workspace_size_for_chunk(T, Hd, V, args.bwd_chunk)
            if bws_bytes == 0:
                raise SystemExit("--bwd-chunk must be a positive multiple of 128")
        self.bws = torch.empty(bws_bytes, dtype=torch.uint8, device=dev)
        self.chunk = flce.flce_backward_chunk_tokens(T, Hd, V, bws_bytes)
        self.outs = self.new_outputs()

    def new_outputs(self):
        torch, T, Hd, V, dev = self.torch, self.inp.T, self.inp.Hd, self.inp.V, self.dev
        return {"loss": torch.empty(T if self.wl.reduction == "none" else 1, dtype=torch.float32, device=dev),
                "lse": torch.empty(T, dtype=torch.float32, device=dev),
                "logp": torch.empty(T, dtype=torch.float32, device=dev),
                "n_valid": torch.empty(1, dtype=torch.int64, device=dev),
                "dH": torch.empty((T, Hd), dtype=torch.bfloat16, device=dev),
                "dW": torch.empty((V, Hd), dtype=torch.float32, device=dev)}

    def step(self, ins, outs):
        H, W, y, dl = ins
        f, ign, red = self.flce, self.inp.ignore_index, self.wl.reduction
        f.flce_forward(H, W, y, ign, red, workspace=self.fws, out=outs)
        f.flce_backward(dl, H, W, y, outs["lse"], ign, red, workspace=self.bws, out=outs)

    def readback(self, outs):
        return [outs["loss"], outs["logp"]]

    def workspaces(self):
        return [self.fws, self.bws]

    def config(self):
        return {"backward_chunk_tokens": self.chunk}

    def dz_block_bytes(self):
        return 2 * self.chunk * ((self.inp.V + 63) // 64 * 64)


class ScorePath:
    """flce_score: per-token logp, lse and greedy token, no loss and no backward
    (2·T·Hd·V FLOPs per step).  Inputs H, W, targets; logp and the greedy token are read back."""

    name = "score"

    def __init__(self, flce, torch, inp, wl, dev, args):
        self.flce, self.torch, self.inp, self.wl, self.dev = flce, torch, inp, wl, dev
        T, Hd, V = inp.T, inp.Hd, inp.V
        self.metric = "scoring tokens/s (per-token logp + lse + greedy token, no backward)"
        self.flops_per_step = 2.0 * T * Hd * V
        self.flops_executed_per_step = self.flops_per_step
        self.host = host_inputs(torch, inp, with_dloss=False)
        self.ins = tuple(t.to(dev) for t in self.host)
        lib = flce.load_library()
        self.ws = torch.empty(max(lib.flce_score_workspace_size(T, Hd, V), 256), dtype=torch.uint8, device=dev)
        self.outs = self.new_outputs()

    def new_outputs(self):
        torch, T, dev = self.torch, self.inp.T, self.dev
        return {"logp": torch.empty(T, dtype=torch.float32, device=dev),
                "lse": torch.empty(T, dtype=torch.float32, device=dev),
                "argmax": torch.empty(T, dtype=torch.int64, device=dev)}

    def step(self, ins, outs):
        H, W, y = ins
        self.flce.flce_score(H, W, y, self.inp.ignore_index, workspace=self.ws, out=outs)

    def readback(self, outs):
        return [outs["logp"], outs["argmax"]]

    def workspaces(self):
        return [self.ws]

    def config(self):
        return {}

    def dz_block_bytes(self):
        return 0


class VocabSplitPath:
    """The vocab-parallel split emulated on one GPU: W's rows cut into `n` equal shards,
    flce_forward_shard per shard, flce_combine_shards, flce_backward_shard per shard
    (8·T·Hd·V FLOPs per step).  Each shard's bf16 dH partial is left for the caller's
    all-reduce, which is not part of the op; inputs and read-back as the loss path."""

    name = "vocab-split"

    def __init__(self, flce, torch, inp, wl, dev, args):
        self.flce, self.torch, self.inp, self.wl, self.dev = flce, torch, inp, wl, dev
        T, Hd, V = inp.T, inp.Hd, inp.V
        n = args.shards
        if n < 1 or V % n:
            raise SystemExit(f"--shards {n} must divide V = {V}")
        self.bounds = [(i * V // n, (i + 1) * V // n) for i in range(n)]
        self.metric = f"fused linear-CE fwd+bwd tokens/s, vocab split over {n} emulated ranks"
        self.flops_per_step = 8.0 * T * Hd * V
        self.flops_executed_per_step = (2.0 * T + 6.0 * kept_rows(inp, wl)) * Hd * V
        self.host = host_inputs(torch, inp, with_dloss=True)
        self.ins = tuple(t.to(dev) for t in self.host)
        lib = flce.load_library()
        Vs = V // n
        self.fws = torch.empty(flce.flce_forward_workspace_size(T, Hd, Vs), dtype=torch.uint8, device=dev)
        self.cws = torch.empty(max(lib.flce_combine_workspace_size(T, n), 256), dtype=torch.uint8, device=dev)
        self.bws = torch.empty(flce.flce_backward_workspace_size(T, Hd, Vs), dtype=torch.uint8, device=dev)
        self.chunk = flce.flce_backward_chunk_tokens(T, Hd, Vs, self.bws.numel())
        self.outs = self.new_outputs()

    def new_outputs(self):
        torch, T, Hd, V, dev = self.torch, self.inp.T, self.inp.Hd, self.inp.V, self.dev
        n = len(self.bounds)
        return {"shard_lse": torch.empty((n, T), dtype=torch.float32, device=dev),
                "shard_zy": torch.empty((n, T), dtype=torch.float32, device=dev),
                "loss": torch.empty(T if self.wl.reduction == "none" else 1, dtype=torch.float32, device=dev),
                "lse": torch.empty(T, dtype=torch.float32, device=dev),
                "logp": torch.empty(T, dtype=torch.float32, device=dev),
                "n_valid": torch.empty(1, dtype=torch.int64, device=dev),
                "dH_partials": torch.empty((n, T, Hd), dtype=torch.bfloat16, device=dev),
                "dW": torch.empty((V, Hd), dtype=torch.float32, device=dev)}

    def step(self, ins, outs):
        H, W, y, dl = ins
        f, ign, red, V = self.flce, self.inp.ignore_index, self.wl.reduction, self.inp.V
        for i, (a, b) in enumerate(self.bounds):
            f.flce_forward_shard(H, W[a:b], y, a, V, ign, workspace=self.fws,
                                 out={"shard_lse": outs["shard_lse"][i], "shard_zy": outs["shard_zy"][i]})
        f.flce_combine_shards(outs["shard_lse"], outs["shard_zy"], y, V, ign, red, workspace=self.cws, out=outs)
        for i, (a, b) in enumerate(self.bounds):
            f.flce_backward_shard(dl, H, W[a:b], y, outs["lse"], a, V, ign, red, workspace=self.bws,
                                  out={"dH": outs["dH_partials"][i], "dW": outs["dW"][a:b]})

    def readback(self, outs):
        return [outs["loss"], outs["logp"]]

    def workspaces(self):
        return [self.fws, self.cws, self.bws]

    def config(self):
        return {"vocab_shards": len(self.bounds), "shard_rows": self.bounds[0][1] - self.bounds[0][0],
                "backward_chunk_tokens": self.chunk}

    def dz_block_bytes(self):
        return 2 * self.chunk * ((self.bounds[0][1] - self.bounds[0][0] + 63) // 64 * 64)


class TrainPath(LossPath):
    """flce_forward_valid + flce_backward: rows with an ignored target skip the forward's
    contraction too (their lse is not computed); what the autograd wrapper runs."""

    name = "train"

    def __init__(self, flce, torch, inp, wl, dev, args):
        super().__init__(flce, torch, inp, wl, dev, args)
        T, Hd, V = inp.T, inp.Hd, inp.V
        self.metric = "fused linear-CE fwd+bwd tokens/s, masked rows skipped in the forward as well"
        n_valid = int(np.count_nonzero(inp.targets != inp.ignore_index))
        self.flops_executed_per_step = (2.0 * n_valid + 6.0 * kept_rows(inp, wl)) * Hd * V
        self.fws = torch.empty(flce.flce_forward_valid_workspace_size(T, Hd, V), dtype=torch.uint8, device=dev)

    def step(self, ins, outs):
        H, W, y, dl = ins
        f, ign, red = self.flce, self.inp.ignore_index, self.wl.reduction
        f.flce_forward_valid(H, W, y, ign, red, workspace=self.fws, out=outs)
        f.flce_backward(dl, H, W, y, outs["lse"], ign, red, workspace=self.bws, out=outs)


class ScoreValidPath(ScorePath):
    """flce_score_valid: scoring over the rows with a valid target only."""

    name = "score-valid"

    def __init__(self, flce, torch, inp, wl, dev, args):
        super().__init__(flce, torch, inp, wl, dev, args)
        T, Hd, V = inp.T, inp.Hd, inp.V
        self.metric = "scoring tokens/s over the rows with a valid target (masked rows skipped)"
        self.flops_executed_per_step = 2.0 * int(np.count_nonzero(inp.targets != inp.ignore_index)) * Hd * V
        lib = flce.load_library()
        self.ws = torch.empty(max(lib.flce_score_valid_workspace_size(T, Hd, V), 256), dtype=torch.uint8,
                              device=dev)

    def step(self, ins, outs):
        H, W, y = ins
        self.flce.flce_score_valid(H, W, y, self.inp.ignore_index, workspace=self.ws, out=outs)


PATHS = {"loss": LossPath, "train": TrainPath, "score": ScorePath, "score-valid": ScoreValidPath,
         "vocab-split": VocabSplitPath}


def kept_rows(inp, wl):
    """Rows the backward contracts: a valid target and a non-zero upstream weight (the
    others have zero dZ rows and are skipped)."""
    valid = inp.targets != inp.ignore_index
    if wl.reduction == "none":
        return int(np.count_nonzero(valid & (inp.dloss != 0)))
    return int(np.count_nonzero(valid)) if float(inp.dloss[0]) != 0.0 else 0


def host_inputs(torch, inp, with_dloss):
    H_h = torch.from_numpy(inp.H_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    W_h = torch.from_numpy(inp.W_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_h = torch.from_numpy(inp.targets).pin_memory()
    if not with_dloss:
        return (H_h, W_h, y_h)
    return (H_h, W_h, y_h, torch.from_numpy(inp.dloss).pin_memory())


def run_ours(args):
    import torch
    import torch.distributed as dist

    import lm_head_linear_gb300 as flce

    world, rank, local = dist_setup()
    if world > 1:
        if torch.cuda.device_count() <= local:
            print(f"bench.py: rank {rank} has local rank {local} but sees {torch.cuda.device_count()} GPUs",
                  file=sys.stderr, flush=True)
            return 2
        torch.cuda.set_device(local)
        # NCCL's communicator lines (rank, nRanks, device) go to the log, however the
        # ranks were started, unless the caller chose NCCL's log level
        if "NCCL_DEBUG" not in os.environ:
            os.environ["NCCL_DEBUG"] = "INFO"
            os.environ.setdefault("NCCL_DEBUG_SUBSYS", "INIT")
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    wl = workload(args.workload)
    inp = generate(wl, seed=rank, T=args.T, Hd=args.Hd, V=args.V)
    T, Hd, V = inp.T, inp.Hd, inp.V
    stream = torch.cuda.current_stream(dev)
    path = PATHS[args.path](flce, torch, inp, wl, dev, args)

    def step():
        path.step(path.ins, path.outs)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def max_over_ranks(x):
        return reduce_max(x, dev)

    # Device memory: the library allocates nothing itself.  The first step loads its module
    # (kernels plus the 32 MiB static scratch of the workspace-free forward); after that the
    # driver's free-memory count must not move, and the caller's buffers are the inputs, the
    # outputs and the workspaces (the [chunk x V] dZ block being the largest).
    barrier()
    free_before = torch.cuda.mem_get_info(dev)[0]
    step()
    barrier()
    free0 = torch.cuda.mem_get_info(dev)[0]
    for _ in range(args.warmup - 1):
        step()
    barrier()
    free1 = torch.cuda.mem_get_info(dev)[0]
    io_bytes = sum(t.numel() * t.element_size() for t in (*path.ins, *path.outs.values()))
    memory = {"logits_copy_bytes": T * V * 2,
              "workspace_bytes": int(sum(w.numel() for w in path.workspaces())),
              "dz_block_bytes": int(path.dz_block_bytes()), "io_bytes": int(io_bytes),
              "torch_peak_allocated_bytes": int(torch.cuda.max_memory_allocated(dev)),
              "module_load_bytes": int(free_before - free0),
              "driver_free_delta_over_warmup_bytes": int(free0 - free1)}
    for ws in path.workspaces():
        st = flce.flce_read_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {st} after the warm-up")

    # ---- device-resident timed region (value); per-kernel events for the roofline.
    # With --graph the step is captured once into a CUDA graph and the timed loop
    # replays it (for launch-bound shapes); the per-kernel events then come from an
    # eager pass of the same number of steps.
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                step()
        stream.wait_stream(cap)
        for _ in range(args.warmup):
            graph.replay()
        barrier()
    def timed_region():
        flce.flce_profile_collect()
        flce.flce_profile_enable(graph is None)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with ClockSampler(dev.index) as sampler:
            barrier()
            ev0.record(stream)
            for _ in range(args.steps):
                if graph is not None:
                    graph.replay()
                else:
                    step()
            ev1.record(stream)
            barrier()
        flce.flce_profile_enable(False)
        if graph is not None:
            flce.flce_profile_enable(True)
            for _ in range(args.steps):
                step()
            flce.flce_profile_enable(False)
        return max_over_ranks(ev0.elapsed_time(ev1)), flce.flce_profile_collect(), sampler.summary()

    # A run whose clocks show a hardware or thermal slowdown, or an SM clock stuck well
    # below its maximum with no reason given (a clock lock left by someone else), is
    # measured once more; the line then reports the second run and the first one's clocks.
    ms_total, kstats, clocks = timed_region()
    if max_over_ranks(1.0 if clocks_rejected(clocks) else 0.0) > 0.0:  # every rank takes the same branch
        first = clocks
        ms_total, kstats, clocks = timed_region()
        clocks = dict(clocks, remeasured_after=first)
    ms_step = ms_total / args.steps
    value = whole_job_tokens_per_s(T * args.steps, world, ms_total)
    gpu_launches = sum(v["launches"] for v in kstats.values())

    # ---- end to end through the public API with host buffers.  Every step copies its
    # inputs (H, W, targets and, with a backward, dloss) in from pinned host memory and
    # reads its result back out (the loss and per-token log p(target); for scoring, log p
    # and the greedy token); gradients stay on the device, where the rest of a training
    # step consumes them.  The copies run on two copy streams (one per direction) and
    # overlap the neighbouring steps' compute through double-buffered device inputs and
    # outputs.
    e2e_steps = max(2, args.steps)
    back_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in path.readback(path.outs)]
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ins = [path.ins, tuple(torch.empty_like(t) for t in path.ins)]
    outs = [path.outs, path.new_outputs()]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def h2d(j):
        with torch.cuda.stream(s_in):
            for dst, src in zip(ins[j], path.host):
                dst.copy_(src, non_blocking=True)
            ev_in[j].record(s_in)

    # Untimed warm-up of the copy path, as the device path gets its warm-up steps: the
    # first copy out of pinned host memory after a long stretch of GPU work ran at
    # 10-50 GB/s on some boxes against ~210 GB/s for the next ones (cause not
    # established; cold address translations of the host pages would fit), a one-off
    # cost that a timed region of a few steps should not carry.
    for j in range(2):
        h2d(j)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_in[j])
            for dst, src in zip(back_h, path.readback(outs[j])):
                dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # the first input copy is timed on its own stream too: its bandwidth tells a run
    # whose host copies are slow (a busy host) from one whose kernels are
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    c0.record(s_in)
    h2d(0)
    c1.record(s_in)
    c2 = torch.cuda.Event(enable_timing=True)
    c3 = torch.cuda.Event(enable_timing=True)
    for i in range(e2e_steps):
        j = i % 2
        if i + 1 < e2e_steps:
            if i >= 1:
                s_in.wait_event(ev_comp[1 - j])  # that input set was last read by step i - 1
            if i + 2 == e2e_steps:
                c2.record(s_in)  # the last step's input copy, timed as well
            h2d(1 - j)
            if i + 2 == e2e_steps:
                c3.record(s_in)
        stream.wait_event(ev_in[j])
        if i >= 2:
            stream.wait_event(ev_out[j])  # that output set was last copied out after step i - 2
        with torch.cuda.stream(stream):
            path.step(ins[j], outs[j])
        ev_comp[j].record(stream)
        s_out.wait_event(ev_comp[j])
        with torch.cuda.stream(s_out):
            for dst, src in zip(back_h, path.readback(outs[j])):
                dst.copy_(src, non_blocking=True)
            ev_out[j].record(s_out)
    stream.wait_event(ev_out[(e2e_steps - 1) % 2])
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1))
    h2d_bytes = sum(t.numel() * t.element_size() for t in path.host)
    d2h_bytes = sum(t.numel() * t.element_size() for t in back_h)
    first_copy_ms = c0.elapsed_time(c1)
    last_copy_ms = c2.elapsed_time(c3)
    e2e = {"value": whole_job_tokens_per_s(T * e2e_steps, world, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(d2h_bytes), "steps": e2e_steps,
           "h2d_gb_per_s_first_copy": (h2d_bytes / first_copy_ms / 1e6) if first_copy_ms > 0 else None,
           "h2d_gb_per_s_last_copy": (h2d_bytes / last_copy_ms / 1e6) if last_copy_ms > 0 else None}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    tflops = world * path.flops_per_step * args.steps / (ms_total / 1000.0) / 1e12
    tflops_exec = world * path.flops_executed_per_step * args.steps / (ms_total / 1000.0) / 1e12
    dom_name, dom = max(kstats.items(), key=lambda kv: kv[1]["total_ms"])
    avg_ms = dom["total_ms"] / dom["launches"]
    ach = (dom["flops"] / dom["launches"]) / (avg_ms / 1000.0) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    traffic = (traffic_from_profiles(dom_name, T, Hd, V, path.config().get("backward_chunk_tokens"),
                                     dom["launches"] / args.steps)
               if args.path == "loss" else None)
    kernels = {k: {"launches": v["launches"], "avg_ms": v["total_ms"] / v["launches"],
                   "share": v["total_ms"] / sum(x["total_ms"] for x in kstats.values()),
                   "tflops": (v["flops"] / (v["total_ms"] / 1000.0) / 1e12) if v["flops"] else None}
               for k, v in sorted(kstats.items())}
    config = {"workload": wl.name if (T, Hd, V) == (wl.T, wl.Hd, wl.V) else f"{wl.name} at T={T} Hd={Hd} V={V}",
              "T": T, "Hd": Hd, "V": V, "reduction": wl.reduction}
    if args.path != "loss":
        config["path"] = args.path
    config.update(path.config())
    config.update({"l2": "inputs larger than L2 (H %.0f MB + W %.0f MB > 129 MB), no flush" % (
                       T * Hd * 2 / 1e6, V * Hd * 2 / 1e6),
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "launch": "cuda graph replay" if args.graph else "eager"})
    line = {
        "metric": path.metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config,
        "tflops": tflops,
        "tflops_executed": tflops_exec,
        "frac_of_bf16_peak": {"burst": tflops_exec / float(peaks.get("bf16_tflops", 1)),
                              "sustained": tflops_exec / peak_sus, "source": peak_src,
                              "flops": "executed: 2*T*Hd*V forward + 6*Hd*V per row the backward contracts"},
        "roofline": {"bound": "tensor", "kernel": dom_name, "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                     "frac": ach / peak, "traffic": traffic,
                     "peak_kind": f"bf16_tflops, burst ({peak_src})",
                     "peak_sustained": peak_sus, "frac_sustained": ach / peak_sus,
                     "algorithmic_flops_per_launch": dom["flops"] / dom["launches"]},
        "kernels": kernels,
        "gpu_launches": int(gpu_launches),
        "e2e": e2e,
        "clocks": clocks,
        "memory": memory,
    }
    if args.path == "loss":
        line["model_tflops_6THV"] = tflops * 6.0 / 8.0
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(inp, budget_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--T", type=int, default=None, help="override the workload's token count (same recipe)")
    ap.add_argument("--Hd", type=int, default=None, help="override the hidden size")
    ap.add_argument("--V", type=int, default=None, help="override the vocabulary size")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true", help="time replays of a CUDA graph of one step")
    ap.add_argument("--path", choices=sorted(PATHS), default="loss",
                    help="loss: flce_forward + flce_backward (the default); train: flce_forward_valid + "
                         "flce_backward; score: flce_score alone; score-valid: flce_score_valid alone; "
                         "vocab-split: the shard entry points over --shards equal vocab shards")
    ap.add_argument("--shards", type=int, default=2, help="vocab shards of --path vocab-split")
    ap.add_argument("--bwd-chunk", type=int, default=0,
                    help="backward token chunk (a multiple of 128; default: the library's default workspace)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus > 1 and world == 1:
        return spawn_self(args)
    if world > 1 and args.gpus != world:
        print(f"bench.py: --gpus {args.gpus} but the launcher started {world} ranks", file=sys.stderr, flush=True)
        return 2
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
