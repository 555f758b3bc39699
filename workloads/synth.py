"""Workload definitions and seeded input generation.

Every workload is drawn host-side with numpy's PCG64 from ``SeedSequence(seed)``
spawned into six child streams, in this order: hidden states, weights, hidden
outliers, targets, ignore mask, per-sequence advantages.  Real-valued draws are
made in float32, scaled in float32, then rounded to bf16 with round-to-nearest-
even.  The bf16 bit patterns are the inputs: the GPU path receives them as
``torch.bfloat16`` tensors, the oracle receives the same values widened exactly
to float64.

The shapes, distributions, target laws and masking rules follow the five
workloads the fused linear cross-entropy is measured on: a tiny case, a medium
case, the 65,536-token x 124,160-vocab example worked through in "Long-Sequence
MoE RL Training: From First Principles to MI300X" section 3, a 131,072-token
long local sequence, and a policy-gradient weighting case.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

IGNORE_INDEX = -100


@dataclasses.dataclass(frozen=True)
class Workload:
    """Recipe of one synthetic workload.

    ``targets`` is ``"uniform"`` (ids uniform in [0, V)) or ``"zipf"`` (bounded
    Zipf over ranks 1..V with p(k) proportional to k**-zipf_s, sampled by
    inverse CDF, token id = rank - 1).  ``ignore_frac`` sets exactly
    round(ignore_frac * T) randomly chosen rows to ``IGNORE_INDEX``;
    ``prefix_frac`` instead masks the first floor(prefix_frac * L) tokens of
    each of the ``n_seq`` sequences of length L = T / n_seq.  ``dloss`` is
    ``"one"`` (scalar upstream gradient 1) or ``"neg_adv_over_T"`` (per-token
    upstream gradient -adv_s / T with adv_s ~ N(0, 1) drawn once per sequence).
    """

    name: str
    T: int
    Hd: int
    V: int
    w_std: float
    targets: str
    reduction: str
    dloss: str = "one"
    zipf_s: float = 1.1
    ignore_frac: float = 0.0
    prefix_frac: float = 0.0
    n_seq: int = 1
    h_outlier_prob: float = 0.0
    h_outlier_scale: float = 20.0
    description: str = ""

    @property
    def flops(self) -> int:
        """Hardware FLOPs of one forward+backward with recompute: 8*T*Hd*V."""
        return 8 * self.T * self.Hd * self.V


WORKLOADS = {
    w.name: w
    for w in (
        Workload(
            name="tiny_T256_H256_V4096",
            T=256, Hd=256, V=4096, w_std=0.02, targets="uniform",
            reduction="mean",
            description="tiny: H~N(0,1), W~N(0,0.02), uniform targets, no ignored rows, mean",
        ),
        Workload(
            name="medium_T8192_H2048_V124160",
            T=8192, Hd=2048, V=124160, w_std=0.02, targets="zipf",
            ignore_frac=0.05, reduction="mean",
            description="medium: Zipf(1.1) targets, 5% ignored rows, mean over valid rows",
        ),
        Workload(
            name="lmhead_T65536_H2048_V124160",
            T=65536, Hd=2048, V=124160, w_std=0.02, targets="zipf",
            ignore_frac=0.02, reduction="mean", h_outlier_prob=0.001,
            description=("65,536 tokens x 124,160 vocab: H~N(0,1) with 0.1% of entries x20, "
                         "Zipf(1.1) targets, 2% ignored rows, mean"),
        ),
        Workload(
            name="long_T131072_H4096_V124160",
            T=131072, Hd=4096, V=124160, w_std=0.015, targets="uniform",
            reduction="sum",
            description="long local sequence: W~N(0,0.015), uniform targets, no ignored rows, sum",
        ),
        Workload(
            name="rlpg_T32768_H2048_V124160",
            T=32768, Hd=2048, V=124160, w_std=0.02, targets="uniform",
            reduction="none", dloss="neg_adv_over_T", prefix_frac=0.3, n_seq=8,
            description=("policy-gradient weighting: 8 sequences x 4096 tokens, first 30% of each "
                         "sequence ignored, per-token upstream gradient -adv/T, reduction none"),
        ),
    )
}


def workload(name: str) -> Workload:
    """Look a workload up by its full name or by its leading word (e.g. ``"tiny"``)."""
    if name in WORKLOADS:
        return WORKLOADS[name]
    hits = [w for k, w in WORKLOADS.items() if k.split("_")[0] == name]
    if len(hits) != 1:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}")
    return hits[0]


@dataclasses.dataclass
class Inputs:
    """One drawn batch.  ``H_bits`` [T, Hd] and ``W_bits`` [V, Hd] are bf16 bit
    patterns (uint16, row-major); ``targets`` [T] int64; ``dloss`` float32 of
    shape [1] (mean / sum) or [T] (none)."""

    workload: Workload
    T: int
    Hd: int
    V: int
    H_bits: np.ndarray
    W_bits: np.ndarray
    targets: np.ndarray
    dloss: np.ndarray
    reduction: str
    ignore_index: int = IGNORE_INDEX

    def H64(self, rows=None) -> np.ndarray:
        return bf16_bits_to_f64(self.H_bits if rows is None else self.H_bits[rows])

    def W64(self, rows=None) -> np.ndarray:
        return bf16_bits_to_f64(self.W_bits if rows is None else self.W_bits[rows])


def inputs_digest(inp: "Inputs") -> str:
    """sha256 over one drawn batch (bf16 bits of H and W, targets, upstream gradient) in a
    fixed order and byte layout: identifies the inputs a stored expected value was made from."""
    import hashlib
    h = hashlib.sha256()
    for a in (inp.H_bits, inp.W_bits, inp.targets.astype("<i8"), inp.dloss.astype("<f4")):
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bits.

    Inputs here are finite, so NaN handling is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns exactly to float64."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def _zipf_targets(rng: np.random.Generator, T: int, V: int, s: float) -> np.ndarray:
    ranks = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    cdf /= cdf[-1]
    u = rng.random(T)
    return np.minimum(np.searchsorted(cdf, u, side="right"), V - 1).astype(np.int64)


def generate(wl: Workload | str, seed: int = 0, T: Optional[int] = None, Hd: Optional[int] = None,
             V: Optional[int] = None, n_seq: Optional[int] = None) -> Inputs:
    """Draw one batch of ``wl``; ``T``/``Hd``/``V``/``n_seq`` override the shape (same recipe)."""
    if isinstance(wl, str):
        wl = workload(wl)
    T = wl.T if T is None else int(T)
    Hd = wl.Hd if Hd is None else int(Hd)
    V = wl.V if V is None else int(V)
    n_seq = wl.n_seq if n_seq is None else int(n_seq)
    r_h, r_w, r_out, r_tgt, r_ign, r_adv = (
        np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(6))

    H = r_h.standard_normal((T, Hd), dtype=np.float32)
    if wl.h_outlier_prob > 0.0:
        mask = r_out.random((T, Hd), dtype=np.float32) < np.float32(wl.h_outlier_prob)
        H[mask] *= np.float32(wl.h_outlier_scale)
        del mask
    H_bits = bf16_bits_from_f32(H)
    del H
    W = r_w.standard_normal((V, Hd), dtype=np.float32)
    W *= np.float32(wl.w_std)
    W_bits = bf16_bits_from_f32(W)
    del W

    if wl.targets == "uniform":
        targets = r_tgt.integers(0, V, size=T, dtype=np.int64)
    elif wl.targets == "zipf":
        targets = _zipf_targets(r_tgt, T, V, wl.zipf_s)
    else:
        raise ValueError(wl.targets)

    if wl.ignore_frac > 0.0:
        n_ign = int(round(wl.ignore_frac * T))
        rows = r_ign.choice(T, size=n_ign, replace=False)
        targets[rows] = IGNORE_INDEX
    if wl.prefix_frac > 0.0:
        if T % n_seq:
            raise ValueError("T must be a multiple of n_seq for prefix masking")
        L = T // n_seq
        n_pre = int(np.floor(wl.prefix_frac * L))
        for s in range(n_seq):
            targets[s * L: s * L + n_pre] = IGNORE_INDEX

    if wl.dloss == "one":
        dloss = np.ones(1, dtype=np.float32)
    elif wl.dloss == "neg_adv_over_T":
        adv = r_adv.standard_normal(n_seq)
        L = T // n_seq
        dloss = (-np.repeat(adv, L) / T).astype(np.float32)
    else:
        raise ValueError(wl.dloss)

    return Inputs(workload=wl, T=T, Hd=Hd, V=V, H_bits=H_bits, W_bits=W_bits,
                  targets=targets, dloss=dloss, reduction=wl.reduction)
