"""Scoring path (per-token logp, lse and greedy token) through the C ABI,
against the fp64 oracle.

The argmax is an integer decided by floating point.  The kernel decides it on
its fp32-accumulated logits; each logit of those carries at most
gamma_K * sum_k |h_k w_k| of accumulation error (K = Hd, gamma_K = K u / (1 - K u),
u = 2^-24; bf16 products are exact in fp32).  Where the oracle's top-2 gap is
larger than twice the row's largest such bound, the two must agree bit-exactly;
elsewhere the kernel's token must be one of the oracle's near-ties.
"""

import numpy as np
import pytest
import torch

import lm_head_linear_gb300 as flce
import oracle
from workloads import generate

from gpu_helpers import TOL_TOKEN, run, to_device

pytestmark = pytest.mark.gpu


def _bound(H64, W64):
    K = H64.shape[1]
    u = 2.0 ** -24
    gamma = K * u / (1 - K * u)
    return 2.0 * gamma * (np.abs(H64) @ np.abs(W64).T).max(axis=1)


def _check_argmax(got, H64, W64):
    idx, gap = oracle.argmax_rows(H64, W64)
    bound = _bound(H64, W64)
    sure = gap > bound
    assert np.array_equal(got[sure], idx[sure])
    Z = oracle.logits(H64, W64)
    for t in np.nonzero(~sure)[0]:
        assert Z[t, got[t]] >= Z[t, idx[t]] - bound[t]
    return int(sure.sum())


CASES = {
    "zipf_T1000_H256_V5000": ("medium", 1000, 256, 5000),
    "outliers_T640_H512_V4097": ("lmhead", 640, 512, 4097),
    "rl_T768_H192_V3001": ("rlpg", 768, 192, 3001),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_score_matches_oracle(case, cuda_device):
    wl, T, Hd, V = CASES[case]
    inp = generate(wl, T=T, Hd=Hd, V=V, n_seq=8 if wl == "rlpg" else None)
    H, W, y, _ = to_device(inp, cuda_device)
    logp, lse, argmax, ws = flce.flce_score(H, W, y, inp.ignore_index)
    assert flce.flce_read_device_status(ws) == 0
    H64, W64 = inp.H64(), inp.W64()
    ref = oracle.forward(H64, W64, inp.targets, inp.ignore_index, "none")
    assert np.max(np.abs(lse.cpu().numpy() - ref.lse)) <= TOL_TOKEN
    assert np.max(np.abs(logp.cpu().numpy() - ref.logp)) <= TOL_TOKEN
    assert np.all(logp.cpu().numpy()[inp.targets == inp.ignore_index] == 0.0)
    n_sure = _check_argmax(argmax.cpu().numpy(), H64, W64)
    assert n_sure > 0.9 * T
    # the same lse and logp as the loss path
    full = run(inp, cuda_device, backward=False)
    assert float((full["lse"] - lse).abs().max().item()) <= 1e-5


def test_argmax_ties_take_the_lowest_id(cuda_device):
    """Only W rows 10 and 3000 are non-zero, both equal to 0.5 in every column: rows with
    a clearly positive sum of H peak at both (lowest id 10), rows with a clearly negative
    sum peak at the thousands of exact zeros (lowest id 0).  Ids 10 and 3000 fall in
    different 256-column tiles and different vocab ranges."""
    inp = generate("tiny", T=400, Hd=128, V=5000)
    Wb = np.zeros_like(inp.W_bits)
    Wb[10] = 0x3F00  # 0.5
    Wb[3000] = 0x3F00
    inp.W_bits = Wb
    H, W, y, _ = to_device(inp, cuda_device)
    _, _, argmax, _ = flce.flce_score(H, W, y, inp.ignore_index)
    got = argmax.cpu().numpy()
    hsum = inp.H64().sum(axis=1)
    pos, neg = hsum > 0.5, hsum < -0.5
    assert pos.sum() > 50 and neg.sum() > 50
    assert np.all(got[pos] == 10)
    assert np.all(got[neg] == 0)


def test_score_full_size_sampled_rows(cuda_device):
    """The 65,536 x 2048 x 124,160 workload: sampled rows' logp, lse and greedy token."""
    inp = generate("lmhead")
    H, W, y, _ = to_device(inp, cuda_device)
    logp, lse, argmax, ws = flce.flce_score(H, W, y, inp.ignore_index)
    assert flce.flce_read_device_status(ws) == 0
    rows = np.unique(np.concatenate([[0, inp.T - 1], np.random.default_rng(5).choice(inp.T, 30, replace=False)]))
    H64, W64 = inp.H64(rows), inp.W64()
    g = oracle.upstream_grad(inp.dloss, inp.targets, inp.V, inp.ignore_index, inp.reduction)
    ref = oracle.sampled_rows(H64, W64, inp.targets[rows], g[rows], inp.ignore_index)
    assert np.max(np.abs(lse.cpu().numpy()[rows] - ref["lse"])) <= TOL_TOKEN
    assert np.max(np.abs(logp.cpu().numpy()[rows] - ref["logp"])) <= TOL_TOKEN
    _check_argmax(argmax.cpu().numpy()[rows], H64, W64)


@pytest.mark.parametrize("case", ["rl_T768_H192_V3001", "zipf_T1000_H256_V5000"])
def test_score_valid_matches_score_on_valid_rows(case, cuda_device):
    """flce_score_valid skips rows with an ignored target: on every other row lse, logp
    and the greedy token are bit-identical to flce_score's; skipped rows read 0, 0, -1."""
    wl, T, Hd, V = CASES[case]
    inp = generate(wl, T=T, Hd=Hd, V=V, n_seq=8 if wl == "rlpg" else None)
    if wl != "rlpg":
        inp.targets[np.random.default_rng(2).random(T) < 0.3] = inp.ignore_index
    H, W, y, _ = to_device(inp, cuda_device)
    logp, lse, amax, _ = flce.flce_score(H, W, y, inp.ignore_index)
    logp_v, lse_v, amax_v, ws = flce.flce_score_valid(H, W, y, inp.ignore_index)
    assert flce.flce_read_device_status(ws) == 0
    valid = torch.from_numpy(inp.targets != inp.ignore_index).to(cuda_device)
    assert 0 < int(valid.sum().item()) < T
    assert torch.equal(lse[valid], lse_v[valid]) and torch.equal(logp[valid], logp_v[valid])
    assert torch.equal(amax[valid], amax_v[valid])
    assert bool((lse_v[~valid] == 0).all().item()) and bool((logp_v[~valid] == 0).all().item())
    assert bool((amax_v[~valid] == -1).all().item())


def test_score_valid_full_size_policy_gradient(cuda_device):
    """32,768 x 2048 x 124,160 with 30 % of every sequence masked."""
    inp = generate("rlpg")
    H, W, y, _ = to_device(inp, cuda_device)
    logp, lse, amax, _ = flce.flce_score(H, W, y, inp.ignore_index)
    logp_v, lse_v, amax_v, ws = flce.flce_score_valid(H, W, y, inp.ignore_index)
    assert flce.flce_read_device_status(ws) == 0
    valid = torch.from_numpy(inp.targets != inp.ignore_index).to(cuda_device)
    assert torch.equal(lse[valid], lse_v[valid]) and torch.equal(logp[valid], logp_v[valid])
    assert torch.equal(amax[valid], amax_v[valid])
