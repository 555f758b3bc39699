"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function checks the oracle against one outside fact: a closed
form, an invariant of the mathematics, a library routine (torch's CPU
cross-entropy and autograd, in fp64), central finite differences, brute force
on tiny inputs, or a figure printed on the pages.  ``test_planted_mistakes``
plants plausible mistakes in the oracle (on the CPU) and shows that every one
of them trips at least one pin.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle.flce_oracle as fo

IGN = -100
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(seed, T=7, Hd=12, V=37, n_ignore=2, scale_w=0.5):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((T, Hd))
    W = rng.standard_normal((V, Hd)) * scale_w
    y = rng.integers(0, V, T)
    if n_ignore:
        y[rng.choice(T, n_ignore, replace=False)] = IGN
    return H, W, y


# ----------------------------------------------------------------------------- pins

def pin_w_zero_closed_form():
    """W = 0: every logit is 0, so lse = ln V exactly, p = 1/V, dH = 0 and
    dW_v = sum_t g_t (1/V - [y_t = v]) h_t."""
    rng = np.random.default_rng(1)
    T, Hd, V = 6, 8, 29
    H = rng.standard_normal((T, Hd))
    W = np.zeros((V, Hd))
    y = rng.integers(0, V, T)
    y[2] = IGN
    f = fo.forward(H, W, y, IGN, "mean")
    assert np.allclose(f.lse, math.log(V), rtol=0, atol=1e-14)
    valid = y != IGN
    assert np.allclose(f.loss_tok[valid], math.log(V), rtol=0, atol=1e-14)
    assert abs(float(f.loss) - math.log(V)) < 1e-14
    assert f.n_valid == T - 1
    dH, dW = fo.backward(1.0, H, W, y, IGN, "mean")
    assert np.array_equal(dH, np.zeros_like(dH))
    g = np.where(valid, 1.0 / (T - 1), 0.0)
    expect = np.zeros((V, Hd))
    for t in range(T):
        for v in range(V):
            expect[v] += g[t] * (1.0 / V - (1.0 if y[t] == v else 0.0)) * H[t]
    assert np.allclose(dW, expect, rtol=0, atol=1e-14)


def pin_vocab_of_one():
    """V = 1: softmax is 1 for the only class, so loss = 0 and every gradient is 0."""
    rng = np.random.default_rng(2)
    H = rng.standard_normal((5, 8))
    W = rng.standard_normal((1, 8))
    y = np.zeros(5, dtype=np.int64)
    f = fo.forward(H, W, y, IGN, "sum")
    assert np.allclose(f.loss_tok, 0.0, atol=1e-14)
    assert np.allclose(f.lse, H @ W[0], atol=1e-12)
    dH, dW = fo.backward(1.0, H, W, y, IGN, "sum")
    assert np.allclose(dH, 0.0, atol=1e-14) and np.allclose(dW, 0.0, atol=1e-14)


def pin_torch_library():
    """Same numbers as torch's own CPU fp64 linear + cross_entropy and its autograd."""
    for red in ("mean", "sum", "none"):
        H, W, y = _rand_case(3 + len(red), T=9, Hd=10, V=23, n_ignore=3)
        rng = np.random.default_rng(11)
        dloss = rng.standard_normal(9) if red == "none" else np.array([1.7])
        Ht = torch.tensor(H, requires_grad=True)
        Wt = torch.tensor(W, requires_grad=True)
        yt = torch.tensor(y)
        out = torch.nn.functional.cross_entropy(
            torch.nn.functional.linear(Ht, Wt), yt, ignore_index=IGN, reduction=red)
        out.backward(torch.tensor(dloss) if red == "none" else torch.tensor(dloss[0]))
        lse_t = torch.logsumexp(torch.tensor(H) @ torch.tensor(W).T, dim=1).numpy()
        # one row block, and blocks of 4 rows (the last one ragged) to exercise the
        # oracle's accumulation across row blocks
        for rb in (256, 4):
            f = fo.forward(H, W, y, IGN, red, row_block=rb)
            assert np.allclose(np.asarray(f.loss), out.detach().numpy(), rtol=1e-13, atol=1e-13)
            assert np.allclose(f.lse, lse_t, rtol=1e-13, atol=1e-13)
            dH, dW = fo.backward(dloss, H, W, y, IGN, red, row_block=rb)
            assert np.allclose(dH, Ht.grad.numpy(), rtol=1e-12, atol=1e-13)
            assert np.allclose(dW, Wt.grad.numpy(), rtol=1e-12, atol=1e-13)


def pin_finite_differences():
    """Gradients agree with central differences of the oracle's own loss
    (T <= 8, Hd <= 16, V <= 64; step 1e-6; relative error <= 1e-6)."""
    for red in ("mean", "none"):
        H, W, y = _rand_case(21, T=6, Hd=9, V=31, n_ignore=1)
        rng = np.random.default_rng(5)
        c = rng.standard_normal(6)
        dloss = c if red == "none" else np.array([1.0])

        def L(Hx, Wx):
            f = fo.forward(Hx, Wx, y, IGN, red)
            return float(np.dot(c, f.loss)) if red == "none" else float(f.loss)

        dH, dW = fo.backward(dloss, H, W, y, IGN, red)
        eps = 1e-6
        num_dH = np.zeros_like(H)
        for idx in np.ndindex(*H.shape):
            Hp, Hm = H.copy(), H.copy()
            Hp[idx] += eps
            Hm[idx] -= eps
            num_dH[idx] = (L(Hp, W) - L(Hm, W)) / (2 * eps)
        num_dW = np.zeros_like(W)
        for idx in np.ndindex(*W.shape):
            Wp, Wm = W.copy(), W.copy()
            Wp[idx] += eps
            Wm[idx] -= eps
            num_dW[idx] = (L(H, Wp) - L(H, Wm)) / (2 * eps)
        for a, n in ((dH, num_dH), (dW, num_dW)):
            rel = np.linalg.norm(a - n) / max(np.linalg.norm(n), 1e-30)
            assert rel <= 1e-6, rel


def pin_brute_force_tiny():
    """Scalar loops with math.exp / math.log on T=4, Hd=3, V=5 (no matmul, no max trick:
    the logits here are small enough not to overflow)."""
    H, W, y = _rand_case(7, T=4, Hd=3, V=5, n_ignore=1)
    T, Hd = H.shape
    V = W.shape[0]
    z = [[sum(H[t][k] * W[v][k] for k in range(Hd)) for v in range(V)] for t in range(T)]
    lse = [math.log(sum(math.exp(z[t][v]) for v in range(V))) for t in range(T)]
    valid = [y[t] != IGN for t in range(T)]
    n = sum(valid)
    loss_tok = [lse[t] - z[t][y[t]] if valid[t] else 0.0 for t in range(T)]
    f = fo.forward(H, W, y, IGN, "mean")
    assert np.allclose(f.lse, lse, rtol=1e-14, atol=1e-14)
    assert np.allclose(f.loss_tok, loss_tok, rtol=1e-14, atol=1e-14)
    assert abs(float(f.loss) - sum(loss_tok) / n) < 1e-14
    g = [1.0 / n if valid[t] else 0.0 for t in range(T)]
    dz = [[g[t] * (math.exp(z[t][v] - lse[t]) - (1.0 if (valid[t] and y[t] == v) else 0.0))
           for v in range(V)] for t in range(T)]
    dH_bf = [[sum(dz[t][v] * W[v][k] for v in range(V)) for k in range(Hd)] for t in range(T)]
    dW_bf = [[sum(dz[t][v] * H[t][k] for t in range(T)) for k in range(Hd)] for v in range(V)]
    dH, dW = fo.backward(1.0, H, W, y, IGN, "mean")
    assert np.allclose(dH, dH_bf, rtol=1e-13, atol=1e-15)
    assert np.allclose(dW, dW_bf, rtol=1e-13, atol=1e-15)


def pin_shift_invariance_and_overflow():
    """W -> W + 1 b^T adds h_t.b to every logit of row t: loss, logp, dH and dW are
    unchanged (dZ rows sum to 0) and lse moves by h_t.b.  With h_t.b near 800 an
    un-shifted exp overflows even fp64, so this also pins the running-max correction
    that section 8 of "Long-Sequence MoE RL Training: From First Principles to
    MI300X" calls load-bearing."""
    H, W, y = _rand_case(8, T=6, Hd=8, V=33, n_ignore=1)
    b = H.mean(axis=0)
    shift = H @ b
    scale = 800.0 / np.abs(shift).max()
    b = b * scale
    Ws = W + b[None, :]
    with np.errstate(over="ignore"):
        assert not np.all(np.isfinite(np.exp(H @ Ws.T)))
    f0 = fo.forward(H, W, y, IGN, "mean")
    f1 = fo.forward(H, Ws, y, IGN, "mean")
    assert np.all(np.isfinite(f1.lse))
    assert np.allclose(f1.lse - H @ b, f0.lse, rtol=0, atol=1e-9)
    assert np.allclose(f1.loss_tok, f0.loss_tok, rtol=0, atol=1e-9)
    d0 = fo.backward(1.0, H, W, y, IGN, "mean")
    d1 = fo.backward(1.0, H, Ws, y, IGN, "mean")
    assert np.allclose(d0[0], d1[0], rtol=0, atol=1e-9)
    assert np.allclose(d0[1], d1[1], rtol=0, atol=1e-9)


def pin_gradient_sums_vanish():
    """Every dZ row sums to 0, so the vocab-sum of dW vanishes: sum_v dW_v = 0."""
    H, W, y = _rand_case(9, T=8, Hd=16, V=64, n_ignore=2)
    dH, dW = fo.backward(1.0, H, W, y, IGN, "sum")
    assert np.allclose(dW.sum(axis=0), 0.0, atol=1e-13)
    assert np.abs(dW).max() > 1e-3


def pin_ignored_rows():
    """Ignored rows: zero loss, exactly-zero dH rows, not counted in N; mean with
    every row ignored is 0 with zero gradients."""
    H, W, y = _rand_case(10, T=8, Hd=6, V=17, n_ignore=3)
    ign = y == IGN
    f = fo.forward(H, W, y, IGN, "mean")
    assert f.n_valid == int((~ign).sum())
    assert np.all(f.loss_tok[ign] == 0.0) and np.all(f.logp[ign] == 0.0)
    dH, dW = fo.backward(1.0, H, W, y, IGN, "mean")
    assert np.all(dH[ign] == 0.0)
    # dropping the ignored rows changes nothing
    f2 = fo.forward(H[~ign], W, y[~ign], IGN, "mean")
    assert abs(float(f.loss) - float(f2.loss)) < 1e-14
    dH2, dW2 = fo.backward(1.0, H[~ign], W, y[~ign], IGN, "mean")
    assert np.allclose(dW, dW2, rtol=0, atol=1e-15)
    yall = np.full_like(y, IGN)
    fa = fo.forward(H, W, yall, IGN, "mean")
    assert float(fa.loss) == 0.0 and fa.n_valid == 0
    dHa, dWa = fo.backward(1.0, H, W, yall, IGN, "mean")
    assert not dHa.any() and not dWa.any()


def pin_reductions_agree():
    """mean = sum / N, and 'none' gives the per-token terms that 'sum' adds up;
    logp = -loss_t on valid rows (log p(target) = z_y - lse)."""
    H, W, y = _rand_case(12, T=8, Hd=6, V=19, n_ignore=2)
    fn = fo.forward(H, W, y, IGN, "none")
    fs = fo.forward(H, W, y, IGN, "sum")
    fm = fo.forward(H, W, y, IGN, "mean")
    assert abs(float(fs.loss) - fn.loss.sum()) < 1e-13
    assert abs(float(fm.loss) - float(fs.loss) / fm.n_valid) < 1e-14
    Z = H @ W.T
    valid = y != IGN
    P = np.exp(Z) / np.exp(Z).sum(axis=1, keepdims=True)
    assert np.allclose(fn.logp[valid], np.log(P[valid, y[valid]]), rtol=1e-13, atol=1e-14)


def pin_permutation_equivariance():
    """Permuting tokens permutes lse / loss / dH and leaves dW unchanged; permuting the
    vocab (and the targets with it) permutes dW rows and leaves the loss unchanged."""
    H, W, y = _rand_case(13, T=8, Hd=6, V=21, n_ignore=2)
    rng = np.random.default_rng(0)
    pt = rng.permutation(8)
    f = fo.forward(H, W, y, IGN, "none")
    fp = fo.forward(H[pt], W, y[pt], IGN, "none")
    assert np.allclose(fp.loss_tok, f.loss_tok[pt], rtol=0, atol=1e-14)
    dH, dW = fo.backward(np.ones(8), H, W, y, IGN, "none")
    dHp, dWp = fo.backward(np.ones(8), H[pt], W, y[pt], IGN, "none")
    assert np.allclose(dHp, dH[pt], atol=1e-14) and np.allclose(dWp, dW, atol=1e-14)
    pv = rng.permutation(21)
    inv = np.argsort(pv)
    yv = np.where(y == IGN, IGN, inv[np.where(y == IGN, 0, y)])
    fv = fo.forward(H, W[pv], yv, IGN, "none")
    assert np.allclose(fv.loss_tok, f.loss_tok, atol=1e-13)
    dHv, dWv = fo.backward(np.ones(8), H, W[pv], yv, IGN, "none")
    assert np.allclose(dWv, dW[pv], atol=1e-14) and np.allclose(dHv, dH, atol=1e-13)


def pin_pages_memory_arithmetic():
    """The dense-logits byte counts printed on the pages (golden fixture)."""
    n = 0
    with open(os.path.join(GOLDEN, "pages_memory_arithmetic.txt"), encoding="utf-8") as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("FACT"):
                expr, val = line.split()[1].split("=")
                assert eval(expr, {}, {}) == int(val), line  # noqa: S307 - fixture arithmetic
                n += 1
                continue
            kv = dict(p.split("=") for p in line.split())
            nbytes = fo.naive_logits_bytes(int(kv["T"]), int(kv["V"]), int(kv["bytes"]), int(kv["copies"]))
            assert round(nbytes / 1e9, 2) == float(kv["GB"]), line
            if "GiB" in kv:
                assert abs(nbytes / 2**30 - float(kv["GiB"])) <= 0.01 + 1e-12, line
            n += 1
    assert n == 8
    assert fo.naive_logits_bytes(65536, 124160, 2) == 16_273_899_520


def pin_sampled_paths():
    """The row-at-a-time and vocab-row helpers agree with the full oracle."""
    H, W, y = _rand_case(14, T=10, Hd=8, V=40, n_ignore=3)
    dloss = np.random.default_rng(3).standard_normal(10)
    f = fo.forward(H, W, y, IGN, "none")
    dH, dW = fo.backward(dloss, H, W, y, IGN, "none")
    g = fo.upstream_grad(dloss, y, 40, IGN, "none")
    rows = np.array([0, 3, 9, 4])
    s = fo.sampled_rows(H[rows], W, y[rows], g[rows], IGN)
    assert np.allclose(s["lse"], f.lse[rows], atol=1e-13)
    assert np.allclose(s["loss_tok"], f.loss_tok[rows], atol=1e-13)
    assert np.allclose(s["dH"], dH[rows], atol=1e-14)
    vr = np.array([0, 5, 39, 17])
    dWr = fo.dW_rows(H, W[vr], y, g, f.lse, vr, token_block=3)
    assert np.allclose(dWr, dW[vr], atol=1e-14)
    t = fo.token_outputs_given_lse(H, W, y, f.lse, IGN, row_block=4)
    assert np.allclose(t["loss_tok"], f.loss_tok, atol=1e-13) and np.allclose(t["logp"], f.logp, atol=1e-13)
    assert np.all(t["logp"][y == IGN] == 0.0)
    # brute force on one valid row: z_y by a Python loop
    r = int(np.nonzero(y != IGN)[0][0])
    zy = sum(H[r][k] * W[y[r]][k] for k in range(8))
    assert abs(t["logp"][r] - (zy - f.lse[r])) < 1e-12


def pin_vocab_shards():
    """Shard partials over a split of the vocabulary: the log-sum-exp of the shards'
    lse is the whole-vocab lse, each valid target logit comes from exactly one shard,
    and the shards' dZ-column blocks give dW (every vocab row lives in one shard)."""
    H, W, y = _rand_case(16, T=9, Hd=8, V=41, n_ignore=2)
    cuts = [0, 13, 29, 41]
    f = fo.forward(H, W, y, IGN, "mean")
    parts = [fo.shard_partials(H, W[a:b], y, a, IGN) for a, b in zip(cuts[:-1], cuts[1:])]
    lses = np.stack([q[0] for q in parts])
    m = lses.max(axis=0)
    assert np.allclose(m + np.log(np.exp(lses - m).sum(axis=0)), f.lse, rtol=0, atol=1e-13)
    zy = np.stack([q[1] for q in parts]).sum(axis=0)
    valid = y != IGN
    Z = H @ W.T
    assert np.allclose(zy[valid], Z[np.nonzero(valid)[0], y[valid]], atol=1e-13)
    assert np.all(zy[~valid] == 0.0)
    owners = sum(((y >= a) & (y < b) & valid).astype(int) for a, b in zip(cuts[:-1], cuts[1:]))
    assert np.array_equal(owners, valid.astype(int))


def pin_argmax():
    """Greedy token: brute force on a tiny case, lowest id among exact ties, and the
    top-2 gap; permuting the vocabulary permutes the answer."""
    H, W, y = _rand_case(17, T=6, Hd=5, V=23, n_ignore=0)
    idx, gap = fo.argmax_rows(H, W)
    for t in range(6):
        z = [sum(H[t][k] * W[v][k] for k in range(5)) for v in range(23)]
        best = max(range(23), key=lambda v: (z[v], -v))
        assert idx[t] == best
        second = max(z[v] for v in range(23) if v != best)
        assert abs(gap[t] - (z[best] - second)) < 1e-12
    W2 = W.copy()
    W2[[4, 17]] = 3.0  # two identical rows far above the rest for rows with a positive sum
    i2, g2 = fo.argmax_rows(H, W2)
    pos = H.sum(axis=1) > 0.5
    assert np.all(i2[pos] == 4) and np.all(g2[pos] == 0.0)
    pv = np.random.default_rng(1).permutation(23)
    i3, _ = fo.argmax_rows(H, W[pv])
    assert np.array_equal(pv[i3], idx)


PINS = [
    pin_w_zero_closed_form, pin_vocab_of_one, pin_torch_library, pin_finite_differences,
    pin_brute_force_tiny, pin_shift_invariance_and_overflow, pin_gradient_sums_vanish,
    pin_ignored_rows, pin_reductions_agree, pin_permutation_equivariance,
    pin_pages_memory_arithmetic, pin_sampled_paths, pin_vocab_shards, pin_argmax,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


def test_target_out_of_range_is_an_error():
    H, W, y = _rand_case(15, T=4, Hd=4, V=9, n_ignore=0)
    y[1] = 9
    with pytest.raises(ValueError):
        fo.forward(H, W, y, IGN, "mean")
    y[1] = -1
    with pytest.raises(ValueError):
        fo.backward(1.0, H, W, y, IGN, "mean")


# ----------------------------------------------------------------------------- planted mistakes

def _backward_with(contract):
    """The oracle's backward with its two contractions replaced by `contract`."""
    def bwd(dloss, H, W, targets, ignore_index=-100, reduction="mean", row_block=256):
        H = np.asarray(H, dtype=np.float64)
        W = np.asarray(W, dtype=np.float64)
        targets = np.asarray(targets, dtype=np.int64)
        g = fo.upstream_grad(dloss, targets, W.shape[0], ignore_index, reduction)
        dH, dW = np.zeros_like(H), np.zeros_like(W)
        for r0 in range(0, H.shape[0], row_block):
            r1 = min(H.shape[0], r0 + row_block)
            Z = fo.logits(H[r0:r1], W)
            dZ = fo._dZ(Z, fo._row_lse(Z), targets[r0:r1], g[r0:r1])
            dW = contract(dZ, H[r0:r1], W, dH, r0, r1, dW)
        return dH, dW
    return bwd


def _mutants():
    real_forward, real_dZ, real_logits, real_row_lse = fo.forward, fo._dZ, fo.logits, fo._row_lse
    real_upstream = fo.upstream_grad

    def dz_no_onehot(Z, lse, targets, g):
        return g[:, None] * np.exp(Z - lse[:, None])

    def dz_wrong_sign(Z, lse, targets, g):
        P = np.exp(Z - lse[:, None])
        rows = np.nonzero(g != 0.0)[0]
        P[rows, targets[rows]] += 1.0
        return g[:, None] * P

    def logits_reversed_vocab(H, W):
        return real_logits(H, W[::-1])

    def lse_no_max(Z):
        return np.log(np.exp(Z).sum(axis=1))

    def lse_forgot_max_add(Z):
        m = Z.max(axis=1)
        return np.log(np.exp(Z - m[:, None]).sum(axis=1))

    def forward_mean_over_T(H, W, targets, ignore_index=-100, reduction="mean", row_block=256):
        r = real_forward(H, W, targets, ignore_index, reduction, row_block)
        if reduction == "mean":
            r.loss = np.float64(r.loss_tok.sum() / len(targets))
        return r

    def forward_logp_sign(H, W, targets, ignore_index=-100, reduction="mean", row_block=256):
        r = real_forward(H, W, targets, ignore_index, reduction, row_block)
        r.logp = r.loss_tok.copy()
        return r

    def upstream_keeps_ignored(dloss, targets, V, ignore_index=-100, reduction="mean"):
        g = real_upstream(dloss, targets, V, ignore_index, reduction)
        g[np.asarray(targets) == ignore_index] = g.max() if g.size else 0.0
        return g

    def dz_scaled_twice(Z, lse, targets, g):
        return real_dZ(Z, lse, targets, g) * 2.0

    def keeps_last_block(dZ, Hb, W, dH, r0, r1, dW):
        dH[r0:r1] = dZ @ W
        return dZ.T @ Hb                      # '=' where the sum needs '+='

    def dW_rows_reversed(dZ, Hb, W, dH, r0, r1, dW):
        dH[r0:r1] = dZ @ W
        return dW + dZ.T @ Hb[::-1]           # token rows paired with the wrong dZ rows

    def dH_vocab_reversed(dZ, Hb, W, dH, r0, r1, dW):
        dH[r0:r1] = dZ @ W[::-1]              # vocab rows paired with the wrong dZ columns
        return dW + dZ.T @ Hb

    return {
        "dZ drops the one-hot term": ("_dZ", dz_no_onehot),
        "dZ adds the one-hot term": ("_dZ", dz_wrong_sign),
        "dZ scaled twice": ("_dZ", dz_scaled_twice),
        "logits against the wrong vocab row": ("logits", logits_reversed_vocab),
        "lse without the running max": ("_row_lse", lse_no_max),
        "lse forgets to add the max back": ("_row_lse", lse_forgot_max_add),
        "mean divides by T, not N": ("forward", forward_mean_over_T),
        "logp with the wrong sign": ("forward", forward_logp_sign),
        "ignored rows keep a gradient": ("upstream_grad", upstream_keeps_ignored),
        "dW keeps only the last row block": ("backward", _backward_with(keeps_last_block)),
        "dW pairs dZ with the wrong token rows": ("backward", _backward_with(dW_rows_reversed)),
        "dH pairs dZ with the wrong vocab rows": ("backward", _backward_with(dH_vocab_reversed)),
    }


@pytest.mark.parametrize("name", sorted(_mutants()))
def test_planted_mistakes(name, monkeypatch):
    attr, fn = _mutants()[name]
    monkeypatch.setattr(fo, attr, fn)
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake: {name}"


def test_planted_mistake_harness_control(monkeypatch):
    """The rebuilt backward used by the gradient mutants, given the right
    contractions, passes every pin: the mutants are caught for their mistakes."""
    def right(dZ, Hb, W, dH, r0, r1, dW):
        dH[r0:r1] = dZ @ W
        return dW + dZ.T @ Hb
    monkeypatch.setattr(fo, "backward", _backward_with(right))
    for pin in PINS:
        pin()
