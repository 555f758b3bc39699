"""Writes the oracle's per-token log-sum-exp of the three largest workloads.

The sampled-vocab-row check of dW needs the row normaliser lse_t of every
token, one fp64 pass over [T x V] logits (2*T*Hd*V multiply-adds: 3.3e13 for
the 65,536-token workload, 1.3e14 for the 131,072 x 4096 one).  That is too
slow to repeat inside the GPU test suite on the machine's host cores, so it is
computed once here, by the oracle alone, and stored:

    python tests/golden/make_lse_golden.py            # all three workloads
    python tests/golden/make_lse_golden.py lmhead     # one of them

Each output file ``lse_<workload>.npz`` holds

* ``lse``        float32 [T]: ``oracle.forward(...).lse`` (fp64, rounded once
                 to float32 for storage; the rounding, <= 1e-6 at lse ~ 12, is
                 far inside the 2e-3 per-token tolerance);
* ``seed``, ``T``, ``Hd``, ``V``: the recipe the inputs were drawn with;
* ``inputs_sha256``: a digest of the drawn inputs (bf16 bits of H and W,
  targets, upstream gradient), which the tests recompute before trusting the
  stored values: a change of the input recipe cannot go unnoticed.

Nothing here touches the CUDA library; only ``oracle/`` and ``workloads/`` are
imported.
"""

from __future__ import annotations

import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from workloads import generate, inputs_digest, workload  # noqa: E402

WORKLOADS = ("lmhead", "long", "rlpg")
SEED = 0


def golden_path(name: str) -> str:
    return os.path.join(HERE, f"lse_{workload(name).name}.npz")


def make(name: str) -> str:
    inp = generate(workload(name), seed=SEED)
    t0 = time.time()
    ref = oracle.forward(inp.H64(), inp.W64(), inp.targets, inp.ignore_index, inp.reduction, row_block=512)
    path = golden_path(name)
    np.savez_compressed(path, lse=ref.lse.astype(np.float32), seed=np.int64(SEED), T=np.int64(inp.T),
                        Hd=np.int64(inp.Hd), V=np.int64(inp.V), inputs_sha256=np.array(inputs_digest(inp)))
    print(f"{path}: T={inp.T} Hd={inp.Hd} V={inp.V} in {time.time() - t0:.0f} s", flush=True)
    return path


if __name__ == "__main__":
    for n in (sys.argv[1:] or WORKLOADS):
        make(n)
