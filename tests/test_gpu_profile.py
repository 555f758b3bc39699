"""The per-kernel timing aid: while enabled, every launch is recorded with its
kind, device time and algorithmic work; the backward's work counts only the
rows it contracts (those with a non-zero upstream weight)."""

import numpy as np
import pytest
import torch

import lm_head_linear_gb300 as flce
from workloads import generate

from gpu_helpers import to_device

pytestmark = pytest.mark.gpu


def test_profile_counts_launches_and_listed_rows(cuda_device):
    T, Hd, V = 1000, 256, 5000
    inp = generate("medium", T=T, Hd=Hd, V=V)
    inp.targets[::4] = inp.ignore_index  # a quarter of the rows skipped by the backward
    H, W, y, dl = to_device(inp, cuda_device)
    ws = flce.flce_backward_workspace_size_for_chunk(T, Hd, V, 256)
    bws = torch.empty(ws, dtype=torch.uint8, device=cuda_device)
    _, lse, _, _, _ = flce.flce_forward(H, W, y, inp.ignore_index, "mean")  # first call: set-up
    torch.cuda.synchronize()
    flce.flce_profile_collect()
    flce.flce_profile_enable(True)
    try:
        _, lse, _, _, _ = flce.flce_forward(H, W, y, inp.ignore_index, "mean")
        flce.flce_backward(dl, H, W, y, lse, inp.ignore_index, "mean", workspace=bws)
    finally:
        flce.flce_profile_enable(False)
    stats = flce.flce_profile_collect()
    n_chunks = -(-T // 256)
    assert stats["fwd_logits_lse"]["launches"] == 1
    assert stats["fwd_finalize"]["launches"] == 1 and stats["fwd_reduce"]["launches"] == 1
    assert stats["bwd_prep"]["launches"] == 1
    for k in ("bwd_gather", "bwd_dz", "bwd_dh_dw"):
        assert stats[k]["launches"] == n_chunks, k
    assert "bwd_scatter" not in stats  # dH rows are written to their tokens by the dH tiles
    assert all(v["total_ms"] > 0 for v in stats.values())
    kept = int(np.count_nonzero(inp.targets != inp.ignore_index))
    assert stats["fwd_logits_lse"]["flops"] == pytest.approx(2.0 * T * Hd * V)
    assert stats["bwd_dz"]["flops"] == pytest.approx(2.0 * kept * Hd * V)
    assert stats["bwd_dh_dw"]["flops"] == pytest.approx(4.0 * kept * Hd * V)
    assert flce.flce_profile_collect() == {}  # collecting clears the records
