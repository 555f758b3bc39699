"""flce_forward + flce_backward captured in one CUDA graph and replayed: the
replays give bit-identical results to eager calls on the same inputs, also
after new inputs are copied into the captured buffers.  (The first call on a
device sets up kernel attributes and must come before any capture.)"""

import numpy as np
import pytest
import torch

import lm_head_linear_gb300 as flce
from workloads import generate

from gpu_helpers import to_device

pytestmark = pytest.mark.gpu


def _buffers(T, Hd, V, dev, reduction):
    out_f = {"loss": torch.empty(T if reduction == "none" else 1, dtype=torch.float32, device=dev),
             "lse": torch.empty(T, dtype=torch.float32, device=dev),
             "logp": torch.empty(T, dtype=torch.float32, device=dev),
             "n_valid": torch.empty(1, dtype=torch.int64, device=dev)}
    out_b = {"dH": torch.empty((T, Hd), dtype=torch.bfloat16, device=dev),
             "dW": torch.empty((V, Hd), dtype=torch.float32, device=dev)}
    fws = torch.empty(max(flce.flce_forward_workspace_size(T, Hd, V), flce.flce_forward_valid_workspace_size(T, Hd, V)),
                      dtype=torch.uint8, device=dev)
    bws = torch.empty(flce.flce_backward_workspace_size(T, Hd, V), dtype=torch.uint8, device=dev)
    return out_f, out_b, fws, bws


def _step(H, W, y, dl, bufs, reduction, forward=None):
    out_f, out_b, fws, bws = bufs
    (forward or flce.flce_forward)(H, W, y, -100, reduction, workspace=fws, out=out_f)
    flce.flce_backward(dl, H, W, y, out_f["lse"], -100, reduction, workspace=bws, out=out_b)


@pytest.mark.parametrize("shape", [("medium", 1000, 256, 5000, "full"), ("tiny", 256, 256, 4096, "full"),
                                   ("medium", 1000, 256, 5000, "valid")])
def test_graph_replay_matches_eager(shape, cuda_device):
    wl, T, Hd, V, fwd = shape
    forward = flce.flce_forward_valid if fwd == "valid" else flce.flce_forward
    a = generate(wl, T=T, Hd=Hd, V=V, seed=1)
    b = generate(wl, T=T, Hd=Hd, V=V, seed=2)
    red = a.reduction
    H, W, y, dl = to_device(a, cuda_device)
    bufs = _buffers(T, Hd, V, cuda_device, red)
    _step(H, W, y, dl, bufs, red, forward)  # first call on the device: set-up outside the capture
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(cuda_device)
    s.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _step(H, W, y, dl, bufs, red, forward)
    torch.cuda.current_stream(cuda_device).wait_stream(s)

    for inp in (b, a, b):
        Hn, Wn, yn, dln = to_device(inp, cuda_device)
        H.copy_(Hn)
        W.copy_(Wn)
        y.copy_(yn)
        dl.copy_(dln)
        g.replay()
        torch.cuda.synchronize()
        got = {k: v.clone() for d in bufs[:2] for k, v in d.items()}
        ref_bufs = _buffers(T, Hd, V, cuda_device, red)
        _step(Hn, Wn, yn, dln, ref_bufs, red, forward)
        torch.cuda.synchronize()
        for d in ref_bufs[:2]:
            for k, v in d.items():
                assert torch.equal(got[k], v), k
        assert flce.flce_read_device_status(bufs[2]) == 0 and flce.flce_read_device_status(bufs[3]) == 0
    assert np.isfinite(float(bufs[0]["loss"][0].item()))
