"""flce_forward_valid: rows with an ignored target are left out of the forward's
contraction.  Against flce_forward on the same inputs: the loss, logp, n_valid and
the lse of valid rows are bit-identical, ignored rows get lse 0, and a backward
fed either lse gives bit-identical gradients; against the oracle, the usual
tolerances."""

import ctypes

import numpy as np
import pytest
import torch

import lm_head_linear_gb300 as flce
import oracle
from workloads import generate

from gpu_helpers import TOL_GRAD, TOL_TOKEN, rel_fro, to_device

pytestmark = pytest.mark.gpu

CASES = [("medium", 1000, 256, 5000, 0.25, "mean"), ("tiny", 333, 320, 777, 0.5, "sum"),
         ("rlpg", 768, 192, 3001, None, "none"), ("medium", 257, 64, 4097, 0.0, "mean")]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}_T{c[1]}_H{c[2]}_V{c[3]}_{c[5]}")
def test_matches_the_full_forward(case, cuda_device):
    wl, T, Hd, V, ign, red = case
    inp = generate(wl, T=T, Hd=Hd, V=V, **({"n_seq": 4} if wl == "rlpg" else {}))
    if ign is not None:
        rng = np.random.default_rng(T)
        inp.targets[rng.random(T) < ign] = inp.ignore_index
    inp.reduction = red
    if red == "none" and wl != "rlpg":
        inp.dloss = np.random.default_rng(1).standard_normal(T).astype(np.float32)
    elif red != "none":
        inp.dloss = np.array([1.3], dtype=np.float32)
    H, W, y, dl = to_device(inp, cuda_device)
    full = flce.flce_forward(H, W, y, inp.ignore_index, red)
    part = flce.flce_forward_valid(H, W, y, inp.ignore_index, red)
    assert flce.flce_read_device_status(part[4]) == 0
    valid = torch.from_numpy(inp.targets != inp.ignore_index).to(cuda_device)
    assert torch.equal(full[0], part[0]) and torch.equal(full[2], part[2]) and torch.equal(full[3], part[3])
    assert torch.equal(full[1][valid], part[1][valid])
    assert bool((part[1][~valid] == 0).all().item())
    g_full = flce.flce_backward(dl, H, W, y, full[1], inp.ignore_index, red)
    g_part = flce.flce_backward(dl, H, W, y, part[1], inp.ignore_index, red)
    assert torch.equal(g_full[0], g_part[0]) and torch.equal(g_full[1], g_part[1])
    ref = oracle.forward(inp.H64(), inp.W64(), inp.targets, inp.ignore_index, red)
    assert np.max(np.abs(part[2].cpu().numpy() - ref.logp)) <= TOL_TOKEN
    v = valid.cpu().numpy()
    assert np.max(np.abs(part[1].cpu().numpy()[v] - ref.lse[v]), initial=0.0) <= TOL_TOKEN
    dH_ref, dW_ref = oracle.backward(inp.dloss, inp.H64(), inp.W64(), inp.targets, inp.ignore_index, red)
    if np.linalg.norm(dH_ref) > 0:
        assert rel_fro(g_part[0].float().cpu().numpy(), dH_ref) <= TOL_GRAD
        assert rel_fro(g_part[1].cpu().numpy(), dW_ref) <= TOL_GRAD


def test_every_row_ignored_and_empty(cuda_device):
    inp = generate("tiny", T=300, Hd=64, V=500)
    inp.targets[:] = inp.ignore_index
    H, W, y, _ = to_device(inp, cuda_device)
    loss, lse, logp, nv, ws = flce.flce_forward_valid(H, W, y, inp.ignore_index, "mean")
    assert flce.flce_read_device_status(ws) == 0
    assert float(loss.item()) == 0.0 and int(nv.item()) == 0
    assert bool((lse == 0).all().item()) and bool((logp == 0).all().item())
    e = torch.empty((0, 64), dtype=torch.bfloat16, device=cuda_device)
    loss, _, _, nv, _ = flce.flce_forward_valid(e, W, torch.empty(0, dtype=torch.int64, device=cuda_device))
    assert float(loss.item()) == 0.0 and int(nv.item()) == 0


def test_target_out_of_range_is_flagged(cuda_device):
    inp = generate("tiny", T=300, Hd=64, V=500)
    inp.targets[7] = 500
    H, W, y, _ = to_device(inp, cuda_device)
    *_, ws = flce.flce_forward_valid(H, W, y, inp.ignore_index, "mean")
    assert flce.flce_read_device_status(ws) == 6


def test_full_size_policy_gradient_workload(cuda_device):
    """32,768 x 2048 x 124,160 with 30 % of every sequence masked: bit-identical to the full
    forward on the valid rows, and the autograd wrapper (which uses it) agrees with the
    explicit calls."""
    inp = generate("rlpg")
    H, W, y, dl = to_device(inp, cuda_device)
    full = flce.flce_forward(H, W, y, inp.ignore_index, inp.reduction)
    part = flce.flce_forward_valid(H, W, y, inp.ignore_index, inp.reduction)
    valid = torch.from_numpy(inp.targets != inp.ignore_index).to(cuda_device)
    assert torch.equal(full[0], part[0]) and torch.equal(full[2], part[2])
    assert torch.equal(full[1][valid], part[1][valid])
    assert flce.flce_read_device_status(part[4]) == 0
    ws = flce.flce_forward_valid_workspace_size(inp.T, inp.Hd, inp.V)
    assert ws <= flce.flce_forward_workspace_size(inp.T, inp.Hd, inp.V) + 8 * inp.T + 2 * inp.T * inp.Hd + (1 << 20)


def test_abi_rejects_before_launch(cuda_device):
    lib = flce.load_library()
    P = ctypes.c_void_p
    assert lib.flce_forward_valid(P(16), P(16), P(16), 10, 64, 50, -100, 1, P(16), P(16), P(16), None, P(256),
                                  16, None) == 4
    assert lib.flce_forward_valid(P(16), P(16), P(20), 10, 64, 50, -100, 1, P(16), P(16), P(16), None, P(256),
                                  1 << 30, None) == 3
