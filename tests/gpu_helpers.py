"""Helpers shared by the GPU parity tests: upload a drawn batch, run the
library through its C ABI, and the tolerance checks."""

import numpy as np
import torch

import lm_head_linear_gb300 as flce

# Tolerances of the parity bar: per-token loss / logp / lse absolute error,
# gradient relative Frobenius error; integers are compared bit-exact.
TOL_TOKEN = 2e-3
TOL_GRAD = 1e-2


def to_device(inp, dev):
    H = torch.from_numpy(inp.H_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    W = torch.from_numpy(inp.W_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    y = torch.from_numpy(inp.targets).to(dev)
    dloss = torch.from_numpy(inp.dloss).to(dev)
    return H, W, y, dloss


def run(inp, dev, bwd_workspace_bytes=None, backward=True):
    H, W, y, dloss = to_device(inp, dev)
    loss, lse, logp, n_valid, fws = flce.flce_forward(H, W, y, inp.ignore_index, inp.reduction)
    out = {"loss": loss, "lse": lse, "logp": logp, "n_valid": n_valid}
    out["fwd_status"] = flce.flce_read_device_status(fws)
    if backward:
        ws = None
        if bwd_workspace_bytes is not None:
            ws = torch.empty(bwd_workspace_bytes, dtype=torch.uint8, device=dev)
        dH, dW, bws = flce.flce_backward(dloss, H, W, y, lse, inp.ignore_index, inp.reduction, workspace=ws)
        out["dH"], out["dW"] = dH, dW
        out["bwd_status"] = flce.flce_read_device_status(bws)
    torch.cuda.synchronize()
    return out


def rel_fro(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / den) if den > 0 else float(np.linalg.norm(got))


def check_token_outputs(out, ref, valid, reduction, rows=None):
    """lse on every row, logp / loss on valid rows (and exact zeros on ignored rows)."""
    lse = out["lse"].cpu().numpy().astype(np.float64)
    logp = out["logp"].cpu().numpy().astype(np.float64)
    if rows is not None:
        lse, logp = lse[rows], logp[rows]
    assert np.max(np.abs(lse - ref["lse"])) <= TOL_TOKEN, np.max(np.abs(lse - ref["lse"]))
    assert np.max(np.abs(logp - ref["logp"])) <= TOL_TOKEN, np.max(np.abs(logp - ref["logp"]))
    assert np.all(logp[~valid] == 0.0)
    if reduction == "none":
        loss = out["loss"].cpu().numpy().astype(np.float64)
        if rows is not None:
            loss = loss[rows]
        assert np.max(np.abs(loss - ref["loss_tok"])) <= TOL_TOKEN
        assert np.all(loss[~valid] == 0.0)
