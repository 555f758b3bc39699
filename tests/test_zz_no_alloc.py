"""The forward entry point that allocates nothing, called through the C ABI.

Some callers cannot allocate device memory where they need the loss (their
framework's allocator owns the device memory, or they run inside an engine
hook that may not allocate).  flce_forward_noalloc serves them with a scratch
array built into the library.  This test checks that it gives the same loss,
lse, logp and n_valid as flce_forward with a caller-provided workspace (within
the parity tolerances, and in fact bit for bit), on two calls in a row that reuse the shared scratch
with different shapes and reductions, and that it rejects a T the scratch
cannot hold.  The file name makes pytest collect it last.
"""

import ctypes

import pytest
import torch

import lm_head_linear_gb300 as flce
from workloads import generate

from gpu_helpers import TOL_TOKEN, to_device

pytestmark = pytest.mark.gpu


def _noalloc(lib, H, W, y, ignore_index, reduction, dev):
    T, Hd = H.shape
    V = W.shape[0]
    red = flce.REDUCTIONS[reduction]
    loss = torch.full((T if red == 0 else 1,), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)
    logp = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)
    n_valid = torch.full((1,), -1, dtype=torch.int64, device=dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    P = ctypes.c_void_p
    st = lib.flce_forward_noalloc(P(H.data_ptr()), P(W.data_ptr()), P(y.data_ptr()), T, Hd, V, ignore_index, red,
                                  P(loss.data_ptr()), P(lse.data_ptr()), P(logp.data_ptr()), P(n_valid.data_ptr()),
                                  P(status.data_ptr()), P(torch.cuda.current_stream(dev).cuda_stream))
    assert st == 0, lib.flce_last_error()
    torch.cuda.synchronize(dev)
    return loss, lse, logp, n_valid, int(status.item())


def test_noalloc_forward_matches_forward_on_two_calls(cuda_device):
    lib = flce.load_library()
    cases = [("medium", 1000, 256, 5000, None), ("rlpg", 768, 192, 3001, 8)]
    for wl, T, Hd, V, n_seq in cases:
        inp = generate(wl, T=T, Hd=Hd, V=V, n_seq=n_seq)
        H, W, y, _ = to_device(inp, cuda_device)
        ref_loss, ref_lse, ref_logp, ref_n, ws = flce.flce_forward(H, W, y, inp.ignore_index, inp.reduction)
        assert flce.flce_read_device_status(ws) == 0
        loss, lse, logp, n_valid, status = _noalloc(lib, H, W, y, inp.ignore_index, inp.reduction, cuda_device)
        assert status == 0
        assert int(n_valid.item()) == int(ref_n.item())
        for got, want in ((loss, ref_loss), (lse, ref_lse), (logp, ref_logp)):
            assert torch.isfinite(got).all()
            assert float((got - want).abs().max().item()) <= TOL_TOKEN
            # the same kernels on the same inputs, in the same order: bit for bit
            assert torch.equal(got, want)


def test_noalloc_forward_reports_device_status_and_rejects_large_T(cuda_device):
    lib = flce.load_library()
    inp = generate("tiny", T=200, Hd=64, V=300)
    inp.targets[3] = 300
    H, W, y, _ = to_device(inp, cuda_device)
    *_, status = _noalloc(lib, H, W, y, inp.ignore_index, inp.reduction, cuda_device)
    assert status == 6
    P = ctypes.c_void_p
    dummy = torch.empty(16, dtype=torch.float32, device=cuda_device)
    ptr = P(dummy.data_ptr())
    st = lib.flce_forward_noalloc(ptr, ptr, ptr, 253952 + 128, 64, 300, -100, 1, ptr, ptr, ptr, None, None, None)
    assert st == 4
    assert b"scratch" in lib.flce_last_error()
