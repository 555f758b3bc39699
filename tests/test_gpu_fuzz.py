"""Seeded sweep of ragged shapes against the full fp64 oracle: T, Hd and V off
the tile grid, all three reductions, random ignore masks, backward workspaces
that force several token chunks, the scoring path and a random vocab split."""

import numpy as np
import pytest
import torch

import lm_head_linear_gb300 as flce
import oracle
from workloads import IGNORE_INDEX, generate

from gpu_helpers import TOL_GRAD, TOL_TOKEN, check_token_outputs, rel_fro, run, to_device

pytestmark = pytest.mark.gpu


def _cases(n=12, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        T = int(rng.integers(1, 1600))
        Hd = int(rng.choice([64, 128, 192, 320, 512]))
        V = int(rng.integers(1, 9000))
        red = ["mean", "sum", "none"][i % 3]
        ign = float(rng.choice([0.0, 0.1, 0.5]))
        chunk = int(rng.choice([0, 128, 384, 1024]))  # 0: the default workspace
        out.append((i, T, Hd, V, red, ign, chunk))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"T{c[1]}_H{c[2]}_V{c[3]}_{c[4]}_ign{c[5]}_chunk{c[6]}")
def test_random_shape(case, cuda_device):
    i, T, Hd, V, red, ign, chunk = case
    inp = generate("tiny", seed=100 + i, T=T, Hd=Hd, V=V)
    rng = np.random.default_rng(7 + i)
    inp.targets[rng.random(T) < ign] = IGNORE_INDEX
    inp.reduction = red
    inp.dloss = (rng.standard_normal(T).astype(np.float32) if red == "none"
                 else np.array([rng.uniform(0.5, 2.0)], dtype=np.float32))
    ws = None
    if chunk and T > 0:
        ws = flce.flce_backward_workspace_size_for_chunk(T, Hd, V, chunk)
        assert flce.flce_backward_chunk_tokens(T, Hd, V, ws) == min(chunk, -(-T // 128) * 128)
    out = run(inp, cuda_device, bwd_workspace_bytes=ws)
    H64, W64 = inp.H64(), inp.W64()
    ref = oracle.forward(H64, W64, inp.targets, IGNORE_INDEX, red)
    valid = inp.targets != IGNORE_INDEX
    assert out["fwd_status"] == 0 and out["bwd_status"] == 0
    assert int(out["n_valid"].item()) == ref.n_valid
    check_token_outputs(out, {"lse": ref.lse, "logp": ref.logp, "loss_tok": ref.loss_tok}, valid, red)
    if red == "mean":
        assert abs(float(out["loss"].item()) - float(ref.loss)) <= TOL_TOKEN
    elif red == "sum":
        # a sum of up to T terms, each within the per-token bound
        assert abs(float(out["loss"].item()) - float(ref.loss)) <= TOL_TOKEN * max(1, ref.n_valid)
    dH_ref, dW_ref = oracle.backward(inp.dloss, H64, W64, inp.targets, IGNORE_INDEX, red)
    if np.linalg.norm(dH_ref) > 0:
        assert rel_fro(out["dH"].float().cpu().numpy(), dH_ref) <= TOL_GRAD
        assert rel_fro(out["dW"].cpu().numpy(), dW_ref) <= TOL_GRAD
    assert np.all(out["dH"].float().cpu().numpy()[~valid] == 0.0)

    # the masked-row forward and scoring give the same numbers on the valid rows
    H, W, y, _ = to_device(inp, cuda_device)
    vmask = torch.from_numpy(valid).to(cuda_device)
    fv = flce.flce_forward_valid(H, W, y, IGNORE_INDEX, red)
    assert flce.flce_read_device_status(fv[4]) == 0
    assert torch.equal(fv[0], out["loss"]) and torch.equal(fv[2], out["logp"])
    assert torch.equal(fv[1][vmask], out["lse"][vmask]) and bool((fv[1][~vmask] == 0).all().item())
    sv = flce.flce_score_valid(H, W, y, IGNORE_INDEX)
    s_full = flce.flce_score(H, W, y, IGNORE_INDEX)
    assert torch.equal(sv[0], s_full[0]) and torch.equal(sv[2][vmask], s_full[2][vmask])

    # scoring path on the same inputs
    logp, lse, argmax, _ = flce.flce_score(H, W, y, IGNORE_INDEX)
    assert np.max(np.abs(logp.cpu().numpy() - ref.logp)) <= TOL_TOKEN
    idx, gap = oracle.argmax_rows(H64, W64)
    sure = gap > 1e-3
    assert np.array_equal(argmax.cpu().numpy()[sure], idx[sure])

    # a random two-way vocab split reproduces the same lse
    if V >= 2:
        cut = int(rng.integers(1, V))
        parts = [flce.flce_forward_shard(H, W[a:b].contiguous(), y, a, V, IGNORE_INDEX)
                 for a, b in ((0, cut), (cut, V))]
        _, lse_c, logp_c, n_c, _ = flce.flce_combine_shards(torch.stack([p[0] for p in parts]),
                                                            torch.stack([p[1] for p in parts]), y, V,
                                                            IGNORE_INDEX, red)
        assert np.max(np.abs(lse_c.cpu().numpy() - ref.lse)) <= TOL_TOKEN
        assert np.max(np.abs(logp_c.cpu().numpy() - ref.logp)) <= TOL_TOKEN
        assert int(n_c.item()) == ref.n_valid
