"""Plain, slow, fp64 CPU oracle of fused linear cross-entropy.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py, never by the product path.

What is computed (source: "Long-Sequence MoE RL Training: From First Principles
to MI300X", section 3 "Linear cross-entropy: don't build a 32 GB tensor to get
a scalar"):

* logits ``Z = H W^T`` over [tokens x vocab];
* per token, cross-entropy through the softmax: ``loss_t = lse_t - z_{t, y_t}``
  with ``lse_t = log sum_v exp(z_{t,v})``, and ``logp_t = -loss_t``;
* the backward needs only ``dZ = softmax(Z) - onehot(y)``, scaled by the
  upstream per-token gradient ``g_t``; it is contracted into ``dH = dZ W`` and
  ``dW = dZ^T H`` (the page writes the weight gradient in its transposed
  orientation, dW^T; the two are the same numbers).

The fused method reaches these same numbers up to rounding order, so the
oracle is the plain definition written out.  The only restructuring is a loop
over independent blocks of token rows (rows are independent by definition) so
that a [T x V] fp64 array is never held for large T; within a row block the
definition is applied as written, with library matmuls as the contraction
steps.  The log-sum-exp subtracts the row maximum before exponentiating: the
same page (section 8, "Through an AMD lens") notes that dropping the running
max overflows.

Readings where the pages are silent (each is listed in the design notes):
* rows with ``target == ignore_index`` contribute zero loss and zero gradient
  and are not counted in N; ``lse`` is still defined on them;
* ``mean`` divides by N = number of valid rows; with N = 0 the loss and every
  gradient are 0;
* a target outside [0, V) that is not ``ignore_index`` is an error;
* reductions: ``mean`` (sum over valid rows / N), ``sum``, ``none`` (per token);
* upstream gradient: ``g_t = dloss / N`` (mean), ``dloss`` (sum),
  ``dloss_t`` (none), and 0 on ignored rows.
"""

from __future__ import annotations

import dataclasses
from typing import Sequence

import numpy as np

REDUCTIONS = ("none", "mean", "sum")


def logits(H: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Z = H W^T (section 3 of the page).  fp64 in, fp64 out."""
    return np.asarray(H, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def valid_mask(targets: np.ndarray, V: int, ignore_index: int) -> np.ndarray:
    """Rows that take part in the loss; raises on an out-of-range target."""
    targets = np.asarray(targets, dtype=np.int64)
    valid = targets != ignore_index
    bad = valid & ((targets < 0) | (targets >= V))
    if bad.any():
        raise ValueError(f"target out of range [0, {V}) at rows {np.nonzero(bad)[0][:8]}")
    return valid


def _row_lse(Z: np.ndarray) -> np.ndarray:
    """lse_t = m_t + log sum_v exp(z_{t,v} - m_t), m_t = max_v z_{t,v}."""
    m = Z.max(axis=1)
    return m + np.log(np.exp(Z - m[:, None]).sum(axis=1))


@dataclasses.dataclass
class ForwardResult:
    lse: np.ndarray          # [T] fp64, defined on every row
    logp: np.ndarray         # [T] fp64, log p(target); 0 on ignored rows
    loss_tok: np.ndarray     # [T] fp64, lse - z_target; 0 on ignored rows
    loss: np.ndarray         # scalar (mean / sum) or [T] (none)
    n_valid: int


def forward(H: np.ndarray, W: np.ndarray, targets: np.ndarray, ignore_index: int = -100,
            reduction: str = "mean", row_block: int = 256) -> ForwardResult:
    """Forward of the linear cross-entropy: loss, lse and logp per token."""
    if reduction not in REDUCTIONS:
        raise ValueError(reduction)
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    T, V = H.shape[0], W.shape[0]
    targets = np.asarray(targets, dtype=np.int64)
    valid = valid_mask(targets, V, ignore_index)
    lse = np.zeros(T)
    zy = np.zeros(T)
    for r0 in range(0, T, row_block):
        r1 = min(T, r0 + row_block)
        Z = logits(H[r0:r1], W)
        lse[r0:r1] = _row_lse(Z)
        rows = np.arange(r1 - r0)
        v = valid[r0:r1]
        zy[r0:r1][v] = Z[rows[v], targets[r0:r1][v]]
    loss_tok = np.where(valid, lse - zy, 0.0)
    logp = -loss_tok
    n_valid = int(valid.sum())
    if reduction == "none":
        loss = loss_tok.copy()
    elif reduction == "sum":
        loss = np.float64(loss_tok.sum())
    else:
        loss = np.float64(loss_tok.sum() / n_valid) if n_valid > 0 else np.float64(0.0)
    return ForwardResult(lse=lse, logp=logp, loss_tok=loss_tok, loss=loss, n_valid=n_valid)


def upstream_grad(dloss, targets: np.ndarray, V: int, ignore_index: int = -100,
                  reduction: str = "mean") -> np.ndarray:
    """Per-token weight g_t of dZ's row t, from the gradient of the reduced loss."""
    valid = valid_mask(targets, V, ignore_index)
    T = valid.shape[0]
    dloss = np.asarray(dloss, dtype=np.float64).reshape(-1)
    if reduction == "none":
        if dloss.shape[0] != T:
            raise ValueError("reduction 'none' takes one upstream gradient per token")
        g = dloss.copy()
    elif reduction == "sum":
        g = np.full(T, dloss[0])
    elif reduction == "mean":
        n = int(valid.sum())
        g = np.full(T, dloss[0] / n if n > 0 else 0.0)
    else:
        raise ValueError(reduction)
    return np.where(valid, g, 0.0)


def _dZ(Z: np.ndarray, lse: np.ndarray, targets: np.ndarray, g: np.ndarray) -> np.ndarray:
    """dZ = g_t * (softmax(Z) - onehot(y)) for one block of rows (section 3 of the page)."""
    P = np.exp(Z - lse[:, None])
    rows = np.nonzero(g != 0.0)[0]
    P[rows, targets[rows]] -= 1.0
    return g[:, None] * P


def backward(dloss, H: np.ndarray, W: np.ndarray, targets: np.ndarray, ignore_index: int = -100,
             reduction: str = "mean", row_block: int = 256):
    """Gradients (dH [T, Hd], dW [V, Hd]) of the reduced loss, fp64.

    The logit rows are recomputed from H and W, as the page's backward does; the
    row normaliser lse comes from the same plain definition as the forward.
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    T, V = H.shape[0], W.shape[0]
    targets = np.asarray(targets, dtype=np.int64)
    g = upstream_grad(dloss, targets, V, ignore_index, reduction)
    dH = np.zeros_like(H)
    dW = np.zeros_like(W)
    for r0 in range(0, T, row_block):
        r1 = min(T, r0 + row_block)
        Z = logits(H[r0:r1], W)
        dZ = _dZ(Z, _row_lse(Z), targets[r0:r1], g[r0:r1])
        dH[r0:r1] = dZ @ W
        dW += dZ.T @ H[r0:r1]
    return dH, dW


def sampled_rows(H_rows: np.ndarray, W: np.ndarray, targets_rows: np.ndarray, g_rows: np.ndarray,
                 ignore_index: int = -100):
    """lse, z_target, loss_t, logp_t and dH_t for a set of token rows, computed one row at a time.

    Every quantity of a token row depends only on that row, so this is the
    full definition restricted to the rows given.  ``g_rows`` is the upstream
    weight of each row (see :func:`upstream_grad`).
    """
    H_rows = np.asarray(H_rows, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    V = W.shape[0]
    targets_rows = np.asarray(targets_rows, dtype=np.int64)
    valid = valid_mask(targets_rows, V, ignore_index)
    n = H_rows.shape[0]
    lse = np.zeros(n)
    loss = np.zeros(n)
    dH = np.zeros_like(H_rows)
    for i in range(n):
        z = W @ H_rows[i]
        lse[i] = _row_lse(z[None, :])[0]
        if valid[i]:
            loss[i] = lse[i] - z[targets_rows[i]]
        dz = _dZ(z[None, :], lse[i:i + 1], targets_rows[i:i + 1],
                 np.asarray([g_rows[i] if valid[i] else 0.0]))
        dH[i] = (dz @ W)[0]
    return {"lse": lse, "loss_tok": loss, "logp": -loss, "dH": dH}


def dW_rows(H: np.ndarray, W_rows: np.ndarray, targets: np.ndarray, g: np.ndarray,
            lse: np.ndarray, vocab_rows: Sequence[int], token_block: int = 8192) -> np.ndarray:
    """dW_v = sum_t dZ_{t,v} h_t for the vocab rows given.

    ``lse`` [T] must be the oracle's own row normaliser for every token (from
    :func:`forward`); ``g`` [T] is the upstream weight from
    :func:`upstream_grad`; ``W_rows`` holds the weight rows of ``vocab_rows``.
    """
    H = np.asarray(H, dtype=np.float64)
    W_rows = np.asarray(W_rows, dtype=np.float64)
    targets = np.asarray(targets, dtype=np.int64)
    vocab_rows = np.asarray(vocab_rows, dtype=np.int64)
    out = np.zeros((len(vocab_rows), H.shape[1]))
    for t0 in range(0, H.shape[0], token_block):
        t1 = min(H.shape[0], t0 + token_block)
        Z = H[t0:t1] @ W_rows.T                       # [tb, nv]
        P = np.exp(Z - lse[t0:t1, None])
        P -= (targets[t0:t1, None] == vocab_rows[None, :])
        dZ = g[t0:t1, None] * P
        out += dZ.T @ H[t0:t1]
    return out


def token_outputs_given_lse(H: np.ndarray, W: np.ndarray, targets: np.ndarray, lse: np.ndarray,
                            ignore_index: int = -100, row_block: int = 8192):
    """Per-token loss_t = lse_t - z_{t, y_t} and logp_t = -loss_t (0 on ignored rows) on every
    row, given the oracle's own row normaliser ``lse`` [T] (from :func:`forward`).

    Only the target logit z_{t, y_t} = h_t . w_{y_t} of each row is formed (T dot products
    of length Hd instead of T x V), so a stored lse turns into the per-token outputs of a
    large batch cheaply.  Same definitions as :func:`forward` (section 3 of the page).
    """
    H = np.asarray(H)
    W = np.asarray(W)
    targets = np.asarray(targets, dtype=np.int64)
    valid = valid_mask(targets, W.shape[0], ignore_index)
    zy = np.zeros(H.shape[0])
    for r0 in range(0, H.shape[0], row_block):
        r1 = min(H.shape[0], r0 + row_block)
        v = valid[r0:r1]
        Hb = np.asarray(H[r0:r1][v], dtype=np.float64)
        Wb = np.asarray(W[targets[r0:r1][v]], dtype=np.float64)
        zy[r0:r1][v] = np.einsum("ij,ij->i", Hb, Wb)
    loss_tok = np.where(valid, np.asarray(lse, dtype=np.float64) - zy, 0.0)
    return {"loss_tok": loss_tok, "logp": -loss_tok}


def shard_partials(H: np.ndarray, W_shard: np.ndarray, targets: np.ndarray, vocab_offset: int,
                   ignore_index: int = -100, row_block: int = 256):
    """Per-row partials of one vocab shard: the log-sum-exp over the shard's logit
    columns, and the target logit where the shard holds the target row (0 elsewhere).

    ``W_shard`` holds global vocab rows [vocab_offset, vocab_offset + V_shard).  The
    shard's lse is the plain definition restricted to its columns; the whole-vocab
    lse is the log-sum-exp of the shards' lse (the vocab-parallel split of the
    Megatron-Lite / bumblebee post, section 2.3 Step 1).
    """
    H = np.asarray(H, dtype=np.float64)
    W_shard = np.asarray(W_shard, dtype=np.float64)
    targets = np.asarray(targets, dtype=np.int64)
    T, Vs = H.shape[0], W_shard.shape[0]
    local = targets - vocab_offset
    owned = (targets != ignore_index) & (local >= 0) & (local < Vs)
    lse = np.zeros(T)
    zy = np.zeros(T)
    for r0 in range(0, T, row_block):
        r1 = min(T, r0 + row_block)
        Z = logits(H[r0:r1], W_shard)
        lse[r0:r1] = _row_lse(Z)
        rows = np.arange(r1 - r0)
        o = owned[r0:r1]
        zy[r0:r1][o] = Z[rows[o], local[r0:r1][o]]
    return lse, zy


def argmax_rows(H: np.ndarray, W: np.ndarray, row_block: int = 256):
    """Greedy token per row: argmax_v z_{t,v} (lowest id on ties) and the gap between
    the largest and the second-largest logit (at another id) of the row."""
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    T, V = H.shape[0], W.shape[0]
    idx = np.zeros(T, dtype=np.int64)
    gap = np.full(T, np.inf)
    for r0 in range(0, T, row_block):
        r1 = min(T, r0 + row_block)
        Z = logits(H[r0:r1], W)
        i = np.argmax(Z, axis=1)
        idx[r0:r1] = i
        if V > 1:
            top = Z[np.arange(r1 - r0), i]
            Z[np.arange(r1 - r0), i] = -np.inf
            gap[r0:r1] = top - Z.max(axis=1)
    return idx, gap


def naive_logits_bytes(T: int, V: int, bytes_per_elem: int, copies: int = 1) -> int:
    """Bytes of ``copies`` dense [T x V] logits tensors (section 3 of the page;
    section 2.3 Step 1 of the Megatron-Lite / bumblebee post)."""
    return int(T) * int(V) * int(bytes_per_elem) * int(copies)


__all__ = [
    "ForwardResult", "argmax_rows", "backward", "dW_rows", "forward", "logits", "naive_logits_bytes",
    "sampled_rows", "shard_partials", "token_outputs_given_lse", "upstream_grad", "valid_mask", "REDUCTIONS",
]

