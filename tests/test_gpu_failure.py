"""Failure detection on the GPU without a fault: a bounded wait that runs out
reports FLCE_ERR_TIMEOUT through the status word, and the context stays usable."""

import time

import numpy as np
import pytest
import torch

import lm_head_linear_gb300 as flce
from workloads import generate

from gpu_helpers import run

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_device):
    t0 = time.perf_counter()
    status = flce.flce_selftest_wait_timeout(20_000_000, device=cuda_device)
    elapsed = time.perf_counter() - t0
    assert status == 7  # FLCE_ERR_TIMEOUT
    assert 0.015 < elapsed < 5.0
    # the context is healthy: a normal call runs and reports no error
    inp = generate("tiny", T=300, Hd=128, V=1000)
    out = run(inp, cuda_device)
    assert out["fwd_status"] == 0 and out["bwd_status"] == 0
    assert np.isfinite(float(out["loss"].item()))
    torch.cuda.synchronize()


def test_selftest_rejects_out_of_range_limits(cuda_device):
    with pytest.raises(flce.FlceError) as e:
        flce.flce_selftest_wait_timeout(10, device=cuda_device)
    assert e.value.status == 1
