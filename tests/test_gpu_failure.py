"""Failure detection on the GPU without a fault: a bounded wait that runs out
reports FLCE_ERR_TIMEOUT through the status word, and the context stays usable."""

import time

import numpy as np
import pytest
import torch

import lm_head_linear_gb300 as flce
from workloads import generate

from gpu_helpers import run, to_device

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


def test_gemm_abort_path_reports_timeout(cuda_device):
    """One 256 x 256 forward tile with K = Hd = 524,288 keeps one SM pair's tensor
    cores busy for ~2 ms.  With the wait limit at 1 ms the epilogue's wait for that
    accumulator runs out inside a legitimate GEMM: the kernel must take its abort path
    (abort flag, drains, TMEM freed), report FLCE_ERR_TIMEOUT and leave the context
    usable.  With the default limit the same shape matches the oracle."""
    import oracle
    from gpu_helpers import TOL_TOKEN
    inp = generate("tiny", T=256, Hd=524288, V=256)
    H, W, y, _ = to_device(inp, cuda_device)
    try:
        flce.flce_set_wait_timeout_ns(1_000_000)
        _, _, _, _, ws = flce.flce_forward(H, W, y)
        assert flce.flce_read_device_status(ws) == 7
    finally:
        flce.flce_set_wait_timeout_ns(4_000_000_000)
    loss, lse, logp, n_valid, ws = flce.flce_forward(H, W, y)
    assert flce.flce_read_device_status(ws) == 0
    # At this K the fp32 tensor-core accumulation (one rounding per K = 16 step, 32,768
    # steps) is no longer inside the per-token tolerance; bound it by one ulp of the
    # row's largest |logit| per step.
    H64, W64 = inp.H64(), inp.W64()
    ref = oracle.forward(H64, W64, inp.targets, inp.ignore_index, "mean")
    zmax = np.abs(oracle.logits(H64, W64)).max(axis=1)
    ulp = 2.0 ** (np.floor(np.log2(zmax)) - 23)
    bound = (inp.Hd / 16) * ulp + TOL_TOKEN
    assert np.all(np.abs(lse.cpu().numpy() - ref.lse) <= bound)
    small = generate("tiny", T=300, Hd=128, V=1000)
    out = run(small, cuda_device)
    assert out["fwd_status"] == 0 and out["bwd_status"] == 0


def test_backward_abort_path_with_wide_dh_tiles_reports_timeout(cuda_device):
    """The dH+dW kernel's abort path, in a 256 x 512 dH tile (both TMEM accumulators,
    the stage ring cut for wide tiles).  T = 256, Hd = 512, V = 400,000: the one wide
    dH tile has a K loop of 6,250 blocks (~3.5 ms of one SM pair) while the other pairs
    run short dW tiles.  With the wait limit at 1 ms the epilogue's wait for that
    tile's accumulators runs out: the call reports FLCE_ERR_TIMEOUT through the status
    word and the context stays usable; with the default limit the same backward
    matches the oracle."""
    import oracle
    from gpu_helpers import TOL_GRAD, rel_fro
    inp = generate("medium", T=256, Hd=512, V=400000)
    H, W, y, dl = to_device(inp, cuda_device)
    _, lse, _, _, fws = flce.flce_forward(H, W, y, inp.ignore_index, inp.reduction)
    assert flce.flce_read_device_status(fws) == 0
    try:
        flce.flce_set_wait_timeout_ns(1_000_000)
        _, _, bws = flce.flce_backward(dl, H, W, y, lse, inp.ignore_index, inp.reduction)
        assert flce.flce_read_device_status(bws) == 7
    finally:
        flce.flce_set_wait_timeout_ns(4_000_000_000)
    dH, dW, bws = flce.flce_backward(dl, H, W, y, lse, inp.ignore_index, inp.reduction)
    assert flce.flce_read_device_status(bws) == 0
    dH_ref, dW_ref = oracle.backward(inp.dloss, inp.H64(), inp.W64(), inp.targets, inp.ignore_index,
                                     inp.reduction, row_block=64)
    assert rel_fro(dH.float().cpu().numpy(), dH_ref) <= TOL_GRAD
    assert rel_fro(dW.cpu().numpy(), dW_ref) <= TOL_GRAD
    small = generate("tiny", T=300, Hd=128, V=1000)
    out = run(small, cuda_device)
    assert out["fwd_status"] == 0 and out["bwd_status"] == 0
