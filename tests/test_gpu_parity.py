"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Element-by-element on shapes the oracle finishes in seconds that span several
128 x 256 tiles and ragged tails; sampled rows and size-independent properties
on the five full-size workloads.
"""

import os

import numpy as np
import pytest
import torch

import lm_head_linear_gb300 as flce
import oracle
from workloads import generate, inputs_digest, workload

from gpu_helpers import TOL_GRAD, TOL_TOKEN, check_token_outputs, rel_fro, run, to_device

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# name -> (workload recipe, T, Hd, V): every case spans several tiles and has ragged edges.
FULL_CASES = {
    "tiny_T256_H256_V4096": ("tiny", None, None, None),
    "zipf_mean_T1000_H256_V5000": ("medium", 1000, 256, 5000),
    "uniform_sum_T333_H320_V777": ("long", 333, 320, 777),
    "rl_none_T768_H192_V3001": ("rlpg", 768, 192, 3001),
    "outliers_T640_H512_V4097": ("lmhead", 640, 512, 4097),
}


def _full_check(inp, out):
    H64, W64 = inp.H64(), inp.W64()
    ref = oracle.forward(H64, W64, inp.targets, inp.ignore_index, inp.reduction)
    valid = inp.targets != inp.ignore_index
    assert out["fwd_status"] == 0 and out["bwd_status"] == 0
    assert int(out["n_valid"].item()) == ref.n_valid
    check_token_outputs(out, {"lse": ref.lse, "logp": ref.logp, "loss_tok": ref.loss_tok}, valid, inp.reduction)
    if inp.reduction != "none":
        assert abs(float(out["loss"].item()) - float(ref.loss)) <= TOL_TOKEN
    dH_ref, dW_ref = oracle.backward(inp.dloss, H64, W64, inp.targets, inp.ignore_index, inp.reduction)
    dH = out["dH"].float().cpu().numpy()
    dW = out["dW"].cpu().numpy()
    assert rel_fro(dH, dH_ref) <= TOL_GRAD, rel_fro(dH, dH_ref)
    assert rel_fro(dW, dW_ref) <= TOL_GRAD, rel_fro(dW, dW_ref)
    assert np.all(dH[~valid] == 0.0)


@pytest.mark.parametrize("case", sorted(FULL_CASES))
def test_full_oracle(case, cuda_device):
    wl, T, Hd, V = FULL_CASES[case]
    inp = generate(wl, T=T, Hd=Hd, V=V, n_seq=8 if wl == "rlpg" else None)
    _full_check(inp, run(inp, cuda_device))


def test_wide_hidden_16384(cuda_device):
    """Hd = 16,384 (1,024 accumulation steps of K = 16 per logit): still inside the
    per-token and gradient tolerances."""
    inp = generate("medium", T=300, Hd=16384, V=2000)
    _full_check(inp, run(inp, cuda_device))


def test_many_token_chunks(cuda_device):
    """A workspace sized for 128-token chunks: dW accumulates over 8 chunks in order."""
    inp = generate("medium", T=1000, Hd=256, V=5000)
    ws = flce.flce_backward_workspace_size(1000, 256, 5000)
    chunk_ws = flce.flce_backward_workspace_size_for_chunk(1000, 256, 5000, 128)
    assert flce.flce_backward_chunk_tokens(1000, 256, 5000, chunk_ws) == 128
    assert chunk_ws < ws
    _full_check(inp, run(inp, cuda_device, bwd_workspace_bytes=chunk_ws))


def test_wide_dh_tiles_odd_block_count_many_chunks(cuda_device):
    """Hd = 1536 (three 512-column dH blocks, 256 x 512 dH tiles) over 128-token chunks:
    each launch cuts its stage ring for the wide tiles and re-cuts it for the dW tiles;
    most SM pairs get no dH tile and start in the dW cut.  Full oracle parity."""
    inp = generate("rlpg", T=1000, Hd=1536, V=3000, n_seq=4)
    chunk_ws = flce.flce_backward_workspace_size_for_chunk(1000, 1536, 3000, 128)
    assert flce.flce_backward_chunk_tokens(1000, 1536, 3000, chunk_ws) == 128
    _full_check(inp, run(inp, cuda_device, bwd_workspace_bytes=chunk_ws))


def test_deterministic(cuda_device):
    inp = generate("medium", T=1000, Hd=256, V=5000)
    a = run(inp, cuda_device)
    b = run(inp, cuda_device)
    for k in ("loss", "lse", "logp", "dH", "dW"):
        assert torch.equal(a[k], b[k]), k


def test_running_max_is_load_bearing(cuda_device):
    """Every logit carries +200 (hidden column 0 = 8, weight column 0 = 25, both exact in
    bf16): exp(z) overflows fp32, the running-max recurrence must not."""
    inp = generate("tiny", T=300, Hd=128, V=1000)
    H = inp.H_bits.copy()
    W = inp.W_bits.copy()
    H[:, 0] = 0x4100  # 8.0
    W[:, 0] = 0x41C8  # 25.0
    inp.H_bits, inp.W_bits = H, W
    out = run(inp, cuda_device)
    assert np.all(np.isfinite(out["lse"].cpu().numpy()))
    assert out["lse"].cpu().numpy().min() > 150.0
    H64, W64 = inp.H64(), inp.W64()
    ref = oracle.forward(H64, W64, inp.targets, inp.ignore_index, inp.reduction)
    valid = inp.targets != inp.ignore_index
    check_token_outputs(out, {"lse": ref.lse, "logp": ref.logp, "loss_tok": ref.loss_tok}, valid, inp.reduction)
    assert abs(float(out["loss"].item()) - float(ref.loss)) <= TOL_TOKEN
    dH_ref, dW_ref = oracle.backward(inp.dloss, H64, W64, inp.targets, inp.ignore_index, inp.reduction)
    dH = out["dH"].float().cpu().numpy()
    assert rel_fro(out["dW"].cpu().numpy(), dW_ref) <= TOL_GRAD
    assert rel_fro(dH[:, 1:], dH_ref[:, 1:]) <= TOL_GRAD
    # dH[:, 0] = 25 * sum_v dZ_tv is 0 exactly; the bf16 storage of dZ (relative rounding
    # <= 2^-9, sum_v |dZ_tv| <= 2 g_t) leaves at most 25 * 2^-8 * g_t there.
    g = oracle.upstream_grad(inp.dloss, inp.targets, inp.V, inp.ignore_index, inp.reduction)
    assert np.all(np.abs(dH[:, 0]) <= 25.0 * 2.0 ** -8 * g + 1e-7)


# ------------------------------------------------------------------ edge cases

def test_vocab_of_one(cuda_device):
    inp = generate("tiny", T=130, Hd=64, V=1)
    out = run(inp, cuda_device)
    _full_check(inp, out)
    assert np.abs(out["loss"].cpu().numpy()).max() <= TOL_TOKEN


def test_all_rows_ignored(cuda_device):
    inp = generate("tiny", T=200, Hd=64, V=300)
    inp.targets[:] = inp.ignore_index
    out = run(inp, cuda_device)
    assert int(out["n_valid"].item()) == 0
    assert float(out["loss"].item()) == 0.0
    assert not out["dH"].float().abs().sum().item() and not out["dW"].abs().sum().item()


def test_single_token_and_empty(cuda_device):
    inp = generate("tiny", T=1, Hd=64, V=700)
    _full_check(inp, run(inp, cuda_device))
    e = generate("tiny", T=0, Hd=64, V=700)
    out = run(e, cuda_device)
    assert float(out["loss"].item()) == 0.0 and int(out["n_valid"].item()) == 0
    assert out["dH"].numel() == 0 and not out["dW"].abs().sum().item()


def test_target_out_of_range_sets_device_status(cuda_device):
    inp = generate("tiny", T=200, Hd=64, V=300)
    inp.targets[5] = 300
    out = run(inp, cuda_device)
    assert out["fwd_status"] == 6 and out["bwd_status"] == 6
    # the bad row is treated as ignored; everything else is still right
    inp.targets[5] = inp.ignore_index
    ok = run(inp, cuda_device)
    assert torch.equal(out["loss"], ok["loss"]) and torch.equal(out["dW"], ok["dW"])


def test_argument_errors(cuda_device):
    inp = generate("tiny", T=64, Hd=64, V=100)
    H, W, y, _ = to_device(inp, cuda_device)
    with pytest.raises(flce.FlceError) as e:
        flce.flce_forward(H, W, y, ignore_index=5)
    assert e.value.status == 1
    with pytest.raises(flce.FlceError) as e:
        flce.flce_forward(H, W, y, workspace=torch.empty(64, dtype=torch.uint8, device=cuda_device))
    assert e.value.status == 4


def test_binding_rejects_buffers_the_library_cannot_use(cuda_device):
    """Buffers the library would write or read through a raw pointer are checked in the
    binding first: a host workspace, an output of the wrong shape or dtype, a host lse."""
    inp = generate("tiny", T=64, Hd=64, V=100)
    H, W, y, dl = to_device(inp, cuda_device)
    with pytest.raises(ValueError):
        flce.flce_forward(H, W, y, workspace=torch.empty(1 << 20, dtype=torch.uint8))
    with pytest.raises(ValueError):
        flce.flce_forward(H, W, y, out={"lse": torch.empty(63, device=cuda_device)})
    with pytest.raises(ValueError):
        flce.flce_forward(H, W, y, out={"n_valid": torch.empty(1, dtype=torch.int32, device=cuda_device)})
    _, lse, _, _, _ = flce.flce_forward(H, W, y)
    with pytest.raises(ValueError):
        flce.flce_backward(dl, H, W, y, lse.cpu())
    with pytest.raises(ValueError):
        flce.flce_backward(dl, H, W, y, lse, out={"dW": torch.empty((100, 64), dtype=torch.bfloat16,
                                                                      device=cuda_device)})
    with pytest.raises(ValueError):
        flce.flce_score(H, W, y, out={"argmax": torch.empty(64, dtype=torch.int32, device=cuda_device)})
    with pytest.raises(ValueError):
        flce.flce_combine_shards(torch.zeros((2, 64), device=cuda_device), torch.zeros((2, 64)), y, 100)
    torch.cuda.synchronize()


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_autograd_wrapper(reduction, cuda_device):
    """linear_cross_entropy through autograd, with a non-trivial upstream gradient for
    each reduction (a scalar for mean / sum, per-token weights for none)."""
    inp = generate("medium", T=300, Hd=128, V=2000)
    H, W, y, _ = to_device(inp, cuda_device)
    Hr = H.clone().requires_grad_(True)
    Wr = W.clone().requires_grad_(True)
    loss = flce.linear_cross_entropy(Hr, Wr, y, reduction=reduction)
    rng = np.random.default_rng(4)
    up = (rng.standard_normal(300) if reduction == "none" else np.array([0.7])).astype(np.float32)
    loss.backward(torch.tensor(up if reduction == "none" else up[0], dtype=torch.float32, device=cuda_device))
    ref = oracle.forward(inp.H64(), inp.W64(), inp.targets, -100, reduction)
    if reduction == "none":
        assert np.max(np.abs(loss.detach().cpu().numpy() - ref.loss_tok)) <= TOL_TOKEN
    else:
        assert abs(float(loss.item()) - float(ref.loss)) <= TOL_TOKEN * (1 if reduction == "mean" else ref.n_valid)
    dH_ref, dW_ref = oracle.backward(up, inp.H64(), inp.W64(), inp.targets, -100, reduction)
    assert rel_fro(Hr.grad.float().cpu().numpy(), dH_ref) <= TOL_GRAD
    assert rel_fro(Wr.grad.float().cpu().numpy(), dW_ref) <= TOL_GRAD


# ------------------------------------------------------------------ the five full-size workloads

FULL_SIZE = ["tiny", "medium", "lmhead", "long", "rlpg"]


@pytest.mark.parametrize("name", FULL_SIZE)
def test_full_size_workload(name, cuda_device):
    """Full-size run in the bench's launch configuration: sampled token rows against the
    oracle (lse, logp, loss, dH), and for dW the properties that hold at any size:
    sum_v dW_v = 0 up to the bf16 rounding of dZ, and <dW, W> = <dH, H>.  On the three
    largest workloads also every token's lse, logp and loss and sampled vocab rows of dW
    (tile and box edges, the most frequent targets, random rows) against the oracle,
    through the oracle's stored lse of the workload (tests/golden/)."""
    wl = workload(name)
    inp = generate(wl)
    torch.cuda.reset_peak_memory_stats(cuda_device)
    base = torch.cuda.memory_allocated(cuda_device)
    out = run(inp, cuda_device)
    peak_extra = torch.cuda.max_memory_allocated(cuda_device) - base
    assert out["fwd_status"] == 0 and out["bwd_status"] == 0
    T, V, Hd = inp.T, inp.V, inp.Hd
    # never a [T x V] buffer.  Everything allocated beyond the inputs and outputs is the two
    # workspaces; the backward one is the [chunk x V] bf16 dZ block plus O(T) scalars, and
    # below one bf16 logits copy whenever T > 256.
    fws_b = flce.flce_forward_workspace_size(T, Hd, V)
    bws_b = flce.flce_backward_workspace_size(T, Hd, V)
    chunk = flce.flce_backward_chunk_tokens(T, Hd, V, bws_b)
    v_pad = (V + 63) // 64 * 64
    # dZ slice [chunk x V], the chunk's H rows [chunk x Hd], g and the row list [T]
    assert bws_b <= 2 * chunk * v_pad + 2 * chunk * Hd + 8 * T + (1 << 20)
    assert fws_b <= (8 * 16 + 4) * (T + 128) + (1 << 20)  # (m, s) per token and vocab range, at most 16 ranges
    io = 2 * T * Hd + 2 * V * Hd + 8 * T + 4 * T + 3 * 4 * T + 8 + 2 * T * Hd + 4 * V * Hd
    assert peak_extra <= io + fws_b + bws_b + (64 << 20)  # caching-allocator rounding
    if T > 256:
        assert bws_b < T * V * 2
    valid = inp.targets != inp.ignore_index
    assert int(out["n_valid"].item()) == int(valid.sum())
    rng = np.random.default_rng(123)
    rows = np.unique(np.concatenate([[0, T - 1], rng.choice(T, size=min(T, 40), replace=False),
                                     np.nonzero(~valid)[0][:4]]))
    W64 = inp.W64()
    g = oracle.upstream_grad(inp.dloss, inp.targets, V, inp.ignore_index, inp.reduction)
    ref = oracle.sampled_rows(inp.H64(rows), W64, inp.targets[rows], g[rows], inp.ignore_index)
    del W64
    check_token_outputs(out, ref, valid[rows], inp.reduction, rows=rows)
    dH = out["dH"].float()
    dH_rows = dH[torch.from_numpy(rows).to(cuda_device)].cpu().numpy()
    assert rel_fro(dH_rows, ref["dH"]) <= TOL_GRAD, rel_fro(dH_rows, ref["dH"])
    assert np.all(dH_rows[~valid[rows]] == 0.0)

    dW = out["dW"]
    H_dev, W_dev = to_device(inp, cuda_device)[:2]
    # (1) sum_v dW_v = sum_t (sum_v dZ_tv) h_t; each stored dZ element carries a relative
    #     rounding error <= 2^-9 and sum_v |dZ_tv| <= 2|g_t|, so |sum_v dW_v| <= 2^-8 sum_t |g_t| |h_t|.
    colsum = dW.double().sum(dim=0).cpu().numpy()
    hnorm = H_dev.float().norm(dim=1).double().cpu().numpy()
    bound = 2.0 ** -8 * float(np.sum(np.abs(g) * hnorm)) + 1e-6
    assert np.linalg.norm(colsum) <= bound, (np.linalg.norm(colsum), bound)
    # (2) <dW, W> = sum_t sum_v dZ_tv z_tv = <dH, H>
    lhs = float((dW.double() * W_dev.double()).sum().item())
    rhs = float((dH.double() * H_dev.double()).sum().item())
    assert abs(lhs - rhs) <= TOL_GRAD * max(abs(lhs), abs(rhs)) + 1e-6, (lhs, rhs)
    assert float(dW.abs().max().item()) > 0.0
    del H_dev, W_dev, dH

    gold = load_lse_golden(wl)
    if gold is not None:
        _check_against_stored_lse(inp, out, gold, g)


def load_lse_golden(wl):
    """The oracle's per-token lse of a full-size workload, stored by
    tests/golden/make_lse_golden.py (None for workloads that have none)."""
    path = os.path.join(GOLDEN, f"lse_{wl.name}.npz")
    if not os.path.exists(path):
        return None
    d = np.load(path)
    return {"lse": d["lse"].astype(np.float64), "seed": int(d["seed"]), "T": int(d["T"]), "Hd": int(d["Hd"]),
            "V": int(d["V"]), "inputs_sha256": str(d["inputs_sha256"])}


def dW_sample_rows(inp, n_random=16, seed=11):
    """Vocab rows for the sampled dW check: both ends, rows on either side of the 64-row
    TMA box, 128-row CTA block and 256-row pair-tile edges (first tiles and last full
    tile), random rows, and the most frequent targets."""
    V = inp.V
    edges = [0, 1, 63, 64, 127, 128, 255, 256, 257, 511, 512]
    last_tile = (V // 256) * 256
    edges += [last_tile - 257, last_tile - 256, last_tile - 1, last_tile, V - 65, V - 64, V - 2, V - 1]
    valid = inp.targets != inp.ignore_index
    counts = np.bincount(inp.targets[valid], minlength=V)
    frequent = np.argsort(-counts, kind="stable")[:4]
    rnd = np.random.default_rng(seed).choice(V, n_random, replace=False)
    rows = np.concatenate([edges, frequent, rnd])
    return np.unique(rows[(rows >= 0) & (rows < V)])


def _check_against_stored_lse(inp, out, gold, g):
    """Every token's lse / logp and sampled vocab rows of dW against the oracle, through
    the oracle's stored lse of this workload (one fp64 pass over T x V, made once)."""
    assert (gold["seed"], gold["T"], gold["Hd"], gold["V"]) == (0, inp.T, inp.Hd, inp.V)
    assert inputs_digest(inp) == gold["inputs_sha256"], "inputs differ from those the stored lse was made from"
    lse_ref = gold["lse"]
    valid = inp.targets != inp.ignore_index
    # per-token outputs on every row (the stored lse is the oracle's; z_y from the inputs)
    lse = out["lse"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse - lse_ref)) <= TOL_TOKEN, np.max(np.abs(lse - lse_ref))
    H64 = inp.H64()
    tok = oracle.token_outputs_given_lse(H64, inp.W64(), inp.targets, lse_ref, inp.ignore_index)
    logp_ref = tok["logp"]
    logp = out["logp"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(logp - logp_ref)) <= TOL_TOKEN, np.max(np.abs(logp - logp_ref))
    assert np.all(logp[~valid] == 0.0)
    if inp.reduction == "none":
        loss = out["loss"].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(loss + logp_ref)) <= TOL_TOKEN
    else:
        loss_ref = float(np.sum(-logp_ref)) / (int(valid.sum()) if inp.reduction == "mean" else 1)
        tol = TOL_TOKEN * (1 if inp.reduction == "mean" else int(valid.sum()))
        assert abs(float(out["loss"].item()) - loss_ref) <= tol, (float(out["loss"].item()), loss_ref)
    # sampled vocab rows of dW
    vr = dW_sample_rows(inp)
    dW_ref = oracle.dW_rows(H64, inp.W64(vr), inp.targets, g, lse_ref, vr)
    dW_rows = out["dW"][torch.from_numpy(vr).to(out["dW"].device)].cpu().numpy().astype(np.float64)
    per_row = [rel_fro(dW_rows[i], dW_ref[i]) for i in range(len(vr))]
    assert rel_fro(dW_rows, dW_ref) <= TOL_GRAD, (rel_fro(dW_rows, dW_ref), max(per_row))
    assert max(per_row) <= TOL_GRAD, dict(zip(vr.tolist(), per_row))


def test_dz_block_beyond_2_31_elements(cuda_device):
    """A backward workspace holding one 8192-token chunk of a 300,001-row vocabulary:
    the dZ block has 8192 x 300,032 = 2.46e9 elements (4.9 GB), past 32-bit element
    offsets.  Sampled token rows against the oracle; dW through the invariants."""
    T, Hd, V = 8192, 64, 300001
    inp = generate("medium", T=T, Hd=Hd, V=V)
    v_pad = (V + 63) // 64 * 64
    ws = flce.flce_backward_workspace_size_for_chunk(T, Hd, V, 8192)
    assert flce.flce_backward_chunk_tokens(T, Hd, V, ws) == 8192 and 8192 * v_pad > 2 ** 31
    out = run(inp, cuda_device, bwd_workspace_bytes=ws)
    assert out["fwd_status"] == 0 and out["bwd_status"] == 0
    valid = inp.targets != inp.ignore_index
    rows = np.unique(np.concatenate([[0, T - 1], np.random.default_rng(9).choice(T, 30, replace=False)]))
    W64 = inp.W64()
    g = oracle.upstream_grad(inp.dloss, inp.targets, V, inp.ignore_index, inp.reduction)
    ref = oracle.sampled_rows(inp.H64(rows), W64, inp.targets[rows], g[rows], inp.ignore_index)
    check_token_outputs(out, ref, valid[rows], inp.reduction, rows=rows)
    dH = out["dH"].float()
    dH_rows = dH[torch.from_numpy(rows).to(cuda_device)].cpu().numpy()
    assert rel_fro(dH_rows, ref["dH"]) <= TOL_GRAD
    H_dev, W_dev = to_device(inp, cuda_device)[:2]
    dW = out["dW"]
    colsum = dW.double().sum(dim=0).cpu().numpy()
    hnorm = H_dev.float().norm(dim=1).double().cpu().numpy()
    assert np.linalg.norm(colsum) <= 2.0 ** -8 * float(np.sum(np.abs(g) * hnorm)) + 1e-6
    lhs = float((dW.double() * W_dev.double()).sum().item())
    rhs = float((dH.double() * H_dev.double()).sum().item())
    assert abs(lhs - rhs) <= TOL_GRAD * max(abs(lhs), abs(rhs)) + 1e-6
    # the last vocab rows (beyond 2^31 / 8192 columns into the block) carry gradient too
    assert float(dW[-64:].abs().max().item()) > 0.0


def test_skipped_rows_do_not_reach_the_gradients(cuda_device):
    """The backward leaves rows whose upstream weight is zero (here: the masked prompt
    prefixes of the policy-gradient recipe, 30 % of every sequence) out of its
    contractions.  With Inf and NaN written into those rows of H, dH and dW are
    bit-identical to the run with the original rows, the skipped rows of dH are exactly
    zero, and both runs match the oracle."""
    inp = generate("rlpg", T=1000, Hd=256, V=5000, n_seq=4)
    H, W, y, dl = to_device(inp, cuda_device)
    ign = torch.from_numpy(inp.targets == inp.ignore_index).to(cuda_device)
    assert 0.2 < float(ign.float().mean().item()) < 0.4
    H_bad = H.clone()
    rows = torch.nonzero(ign).flatten()
    H_bad[rows[0::2]] = float("inf")
    H_bad[rows[1::2]] = float("nan")
    outs = []
    for Hx in (H, H_bad):
        _, lse, _, _, _ = flce.flce_forward(Hx, W, y, inp.ignore_index, inp.reduction)
        dH, dW, ws = flce.flce_backward(dl, Hx, W, y, lse, inp.ignore_index, inp.reduction)
        assert flce.flce_read_device_status(ws) == 0
        outs.append((dH, dW))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert bool((outs[1][0][ign] == 0).all().item())
    assert bool(torch.isfinite(outs[1][1]).all().item())
    dH_ref, dW_ref = oracle.backward(inp.dloss, inp.H64(), inp.W64(), inp.targets, inp.ignore_index, inp.reduction)
    assert rel_fro(outs[1][0].float().cpu().numpy(), dH_ref) <= TOL_GRAD
    assert rel_fro(outs[1][1].cpu().numpy(), dW_ref) <= TOL_GRAD


def test_zero_upstream_gradient_everywhere(cuda_device):
    """Reduction none with dloss = 0 on every row: no row is left for the contractions,
    and dH and dW come out exactly zero (dW from the first chunk's zero fill)."""
    inp = generate("medium", T=700, Hd=128, V=3000)
    H, W, y, _ = to_device(inp, cuda_device)
    _, lse, _, _, _ = flce.flce_forward(H, W, y, inp.ignore_index, "none")
    dW = torch.full((3000, 128), 7.0, device=cuda_device)
    dH = torch.full((700, 128), 7.0, dtype=torch.bfloat16, device=cuda_device)
    _, _, ws = flce.flce_backward(torch.zeros(700, device=cuda_device), H, W, y, lse, inp.ignore_index, "none",
                                  out={"dH": dH, "dW": dW})
    assert flce.flce_read_device_status(ws) == 0
    assert bool((dH == 0).all().item()) and bool((dW == 0).all().item())


def test_full_size_sampled_dW_medium(cuda_device):
    """Sampled vocab rows of dW at the full medium size (T=8192, Hd=2048, V=124,160) against
    the oracle; needs the oracle's lse on every token (one fp64 pass over T x V)."""
    inp = generate("medium")
    out = run(inp, cuda_device)
    H64, W64 = inp.H64(), inp.W64()
    ref = oracle.forward(H64, W64, inp.targets, inp.ignore_index, inp.reduction, row_block=512)
    g = oracle.upstream_grad(inp.dloss, inp.targets, inp.V, inp.ignore_index, inp.reduction)
    rng = np.random.default_rng(7)
    vr = np.unique(np.concatenate([[0, 1, inp.V - 1], rng.choice(inp.V, 29, replace=False),
                                   inp.targets[inp.targets >= 0][:4]]))
    dW_ref = oracle.dW_rows(H64, W64[vr], inp.targets, g, ref.lse, vr)
    dW_rows = out["dW"][torch.from_numpy(vr).to(cuda_device)].cpu().numpy()
    assert rel_fro(dW_rows, dW_ref) <= TOL_GRAD, rel_fro(dW_rows, dW_ref)
    lse = out["lse"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse - ref.lse)) <= TOL_TOKEN
    assert abs(float(out["loss"].item()) - float(ref.loss)) <= TOL_TOKEN


def test_gradient_through_logp(cuda_device):
    """A policy-gradient objective built from the per-token log-probabilities,
    J = -(adv * logp).sum() + 0.3 * loss_mean, differentiated by autograd through
    both outputs; the oracle gets the equivalent per-token weights
    g_t = 0.3 / N + adv_t on valid rows (since logp_t = -loss_t there)."""
    inp = generate("rlpg", T=768, Hd=192, V=3001, n_seq=8)
    H, W, y, _ = to_device(inp, cuda_device)
    adv = torch.from_numpy(np.random.default_rng(3).standard_normal(768).astype(np.float32)).to(cuda_device)
    Hr = H.clone().requires_grad_(True)
    Wr = W.clone().float().requires_grad_(True)
    loss, logp = flce.LinearCrossEntropy.apply(Hr, Wr.to(torch.bfloat16), y, -100, "mean")
    J = -(adv * logp).sum() + 0.3 * loss
    J.backward()
    valid = inp.targets != inp.ignore_index
    n = int(valid.sum())
    g = np.where(valid, 0.3 / n + adv.cpu().numpy().astype(np.float64), 0.0)
    dH_ref, dW_ref = oracle.backward(g, inp.H64(), inp.W64(), inp.targets, inp.ignore_index, "none")
    assert rel_fro(Hr.grad.float().cpu().numpy(), dH_ref) <= TOL_GRAD
    assert rel_fro(Wr.grad.float().cpu().numpy(), dW_ref) <= TOL_GRAD
    lp = flce.linear_log_probs(H, W, y)
    ref = oracle.forward(inp.H64(), inp.W64(), inp.targets, inp.ignore_index, "none")
    assert np.max(np.abs(lp.detach().cpu().numpy() - ref.logp)) <= TOL_TOKEN


def test_paired_torch_baseline(cuda_device):
    """The pages' paired-baseline check: swap the primitive, keep the inputs.  The same
    bf16 inputs through PyTorch's own materialised fp32 logits, cross_entropy and
    autograd on the GPU give the same loss, per-token logp and gradients within the
    tolerances (the oracle is the reference everywhere else)."""
    import torch.nn.functional as F

    inp = generate("medium", T=4096, Hd=1024, V=32000)
    H, W, y, _ = to_device(inp, cuda_device)
    Hf = H.float().requires_grad_(True)
    Wf = W.float().requires_grad_(True)
    z = Hf @ Wf.T
    ref_loss = F.cross_entropy(z, y, ignore_index=inp.ignore_index, reduction="mean")
    ref_loss.backward()
    ref_logp = torch.where(y == inp.ignore_index, torch.zeros_like(z[:, 0]),
                           -F.cross_entropy(z.detach(), y.clamp(min=0), reduction="none"))
    loss, logp = flce.LinearCrossEntropy.apply(H.clone().requires_grad_(True), W, y, inp.ignore_index, "mean")
    assert abs(float(loss.item()) - float(ref_loss.item())) <= TOL_TOKEN
    assert float((logp - ref_logp).abs().max().item()) <= TOL_TOKEN
    dH, dW, _ = flce.flce_backward(torch.ones(1, device=cuda_device), H, W, y,
                                   flce.flce_forward(H, W, y, inp.ignore_index)[1], inp.ignore_index, "mean")
    assert rel_fro(dH.float().cpu().numpy(), Hf.grad.double().cpu().numpy()) <= TOL_GRAD
    assert rel_fro(dW.cpu().numpy(), Wf.grad.double().cpu().numpy()) <= TOL_GRAD
