"""Vocab-parallel split on one GPU: per-shard forward, cross-shard combine and
per-shard backward through the C ABI, against the fp64 oracle and against the
unsharded path.  The shards play the vocab-parallel ranks; summing the dH
partials stands in for the ranks' all-reduce."""

import numpy as np
import pytest
import torch

import lm_head_linear_gb300 as flce
import oracle
from workloads import generate

from gpu_helpers import TOL_GRAD, TOL_TOKEN, rel_fro, run, to_device

pytestmark = pytest.mark.gpu


def _sharded(inp, cuts, dev):
    H, W, y, dloss = to_device(inp, dev)
    lses, zys = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        sl, sz, ws = flce.flce_forward_shard(H, W[a:b].contiguous(), y, a, inp.V, inp.ignore_index)
        assert flce.flce_read_device_status(ws) == 0
        lses.append(sl)
        zys.append(sz)
    shard_lse = torch.stack(lses)
    shard_zy = torch.stack(zys)
    loss, lse, logp, n_valid, cws = flce.flce_combine_shards(shard_lse, shard_zy, y, inp.V, inp.ignore_index,
                                                             inp.reduction)
    assert flce.flce_read_device_status(cws) == 0
    dH = torch.zeros(H.shape, dtype=torch.float32, device=dev)
    dWs = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        dHp, dWp, bws = flce.flce_backward_shard(dloss, H, W[a:b].contiguous(), y, lse, a, inp.V, inp.ignore_index,
                                                 inp.reduction)
        assert flce.flce_read_device_status(bws) == 0
        dH += dHp.float()
        dWs.append(dWp)
    torch.cuda.synchronize()
    return {"shard_lse": shard_lse, "shard_zy": shard_zy, "loss": loss, "lse": lse, "logp": logp,
            "n_valid": n_valid, "dH": dH, "dW": torch.cat(dWs)}


CASES = {
    # three uneven shards, one of them narrower than a 256-column tile at its end
    "three_shards_T1000_H256_V5000": ("medium", 1000, 256, 5000, [0, 2048, 3500, 5000]),
    # the pages' split: a 248,320-row vocabulary over two ranks of 124,160 rows each
    "two_ranks_T512_H256_V248320": ("lmhead", 512, 256, 248320, [0, 124160, 248320]),
    "policy_gradient_none_T768_H192_V3001": ("rlpg", 768, 192, 3001, [0, 1000, 2001, 3001]),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_sharded_matches_oracle_and_unsharded(case, cuda_device):
    wl, T, Hd, V, cuts = CASES[case]
    inp = generate(wl, T=T, Hd=Hd, V=V, n_seq=8 if wl == "rlpg" else None)
    out = _sharded(inp, cuts, cuda_device)
    H64, W64 = inp.H64(), inp.W64()
    valid = inp.targets != inp.ignore_index
    # per-shard partials against the oracle's
    for r, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        ref_lse, ref_zy = oracle.shard_partials(H64, W64[a:b], inp.targets, a, inp.ignore_index)
        assert np.max(np.abs(out["shard_lse"][r].cpu().numpy() - ref_lse)) <= TOL_TOKEN
        assert np.max(np.abs(out["shard_zy"][r].cpu().numpy() - ref_zy)) <= TOL_TOKEN
    ref = oracle.forward(H64, W64, inp.targets, inp.ignore_index, inp.reduction)
    assert int(out["n_valid"].item()) == ref.n_valid
    assert np.max(np.abs(out["lse"].cpu().numpy() - ref.lse)) <= TOL_TOKEN
    assert np.max(np.abs(out["logp"].cpu().numpy() - ref.logp)) <= TOL_TOKEN
    assert np.max(np.abs(np.asarray(out["loss"].cpu().numpy(), np.float64) - np.asarray(ref.loss))) <= TOL_TOKEN
    dH_ref, dW_ref = oracle.backward(inp.dloss, H64, W64, inp.targets, inp.ignore_index, inp.reduction)
    assert rel_fro(out["dH"].cpu().numpy(), dH_ref) <= TOL_GRAD
    assert rel_fro(out["dW"].cpu().numpy(), dW_ref) <= TOL_GRAD
    assert np.all(out["dH"].cpu().numpy()[~valid] == 0.0)
    # and against the unsharded path on the same inputs
    full = run(inp, cuda_device)
    assert float((out["lse"] - full["lse"]).abs().max().item()) <= TOL_TOKEN
    assert rel_fro(out["dW"].cpu().numpy(), full["dW"].cpu().numpy()) <= TOL_GRAD


def test_single_shard_is_the_forward(cuda_device):
    inp = generate("tiny", T=300, Hd=128, V=1000)
    out = _sharded(inp, [0, 1000], cuda_device)
    full = run(inp, cuda_device)
    assert float((out["lse"] - full["lse"]).abs().max().item()) <= 1e-5
    assert float((out["loss"] - full["loss"]).abs().max().item()) <= 1e-5
    assert torch.equal(out["n_valid"], full["n_valid"])


def test_shard_argument_errors(cuda_device):
    inp = generate("tiny", T=64, Hd=64, V=100)
    H, W, y, _ = to_device(inp, cuda_device)
    with pytest.raises(flce.FlceError) as e:
        flce.flce_forward_shard(H, W[:60].contiguous(), y, 50, 100)  # shard [50, 110) leaves [0, 100)
    assert e.value.status == 1
    with pytest.raises(flce.FlceError) as e:
        flce.flce_forward_shard(H, W[:60].contiguous(), y, 0, 100, ignore_index=99)
    assert e.value.status == 1
