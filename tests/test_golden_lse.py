"""The stored oracle lse of the three largest workloads (tests/golden/lse_*.npz).

The files are written by tests/golden/make_lse_golden.py from the oracle alone.
Here, without a GPU: every file is present and names the recipe of its
workload, and for the policy-gradient workload (the smallest, drawn in a few
seconds) the inputs still hash to the stored digest and a handful of stored
rows agree with the oracle's row-at-a-time lse.
"""

import os

import numpy as np
import pytest

import oracle
from workloads import generate, inputs_digest, workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("name", ["lmhead", "long", "rlpg"])
def test_stored_lse_present_and_named(name):
    wl = workload(name)
    d = np.load(os.path.join(GOLDEN, f"lse_{wl.name}.npz"))
    assert (int(d["seed"]), int(d["T"]), int(d["Hd"]), int(d["V"])) == (0, wl.T, wl.Hd, wl.V)
    lse = d["lse"]
    assert lse.shape == (wl.T,) and lse.dtype == np.float32 and np.all(np.isfinite(lse))
    # lse_t >= max_v z_tv > -inf and lse_t <= max_v z_tv + ln V: a loose range check
    assert float(lse.min()) > np.log(wl.V) - 50.0 and float(lse.max()) < np.log(wl.V) + 500.0
    assert len(str(d["inputs_sha256"])) == 64


def test_stored_lse_matches_oracle_rows():
    wl = workload("rlpg")
    d = np.load(os.path.join(GOLDEN, f"lse_{wl.name}.npz"))
    inp = generate(wl, seed=int(d["seed"]))
    assert inputs_digest(inp) == str(d["inputs_sha256"])
    rows = np.array([0, 1, 1228, 4095, 4096, 20000, wl.T - 1])
    g = np.zeros(len(rows))
    ref = oracle.sampled_rows(inp.H64(rows), inp.W64(), np.full(len(rows), -100), g, -100)
    assert np.max(np.abs(d["lse"][rows].astype(np.float64) - ref["lse"])) <= 2e-6
