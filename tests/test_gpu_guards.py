"""Out-of-bounds write checks without a sanitizer: every output and workspace of
every entry point sits inside a larger buffer whose margins hold a byte
pattern; after the call, on ragged shapes, the margins must be untouched."""

import ctypes

import numpy as np
import pytest
import torch

import lm_head_linear_gb300 as flce
from workloads import IGNORE_INDEX, generate

from gpu_helpers import to_device

pytestmark = pytest.mark.gpu

GUARD = 4096       # bytes of margin on each side (a multiple of 256 keeps the alignment)
PATTERN = 0xA5


class Guarded:
    """A device tensor of `shape`/`dtype` with PATTERN-filled margins around it."""

    def __init__(self, shape, dtype, dev):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.nbytes = n
        self.raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device=dev)
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape) if n else \
            torch.empty(shape, dtype=dtype, device=dev)

    def intact(self):
        lo = self.raw[:GUARD]
        hi = self.raw[GUARD + self.nbytes:]
        return bool((lo == PATTERN).all().item()) and bool((hi == PATTERN).all().item())


P = ctypes.c_void_p


def _p(g):
    return P(g.t.data_ptr())


SHAPES = [(333, 320, 777), (1000, 256, 5000), (1, 64, 1), (640, 512, 4097)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"T{s[0]}_H{s[1]}_V{s[2]}")
def test_no_write_outside_any_buffer(shape, cuda_device):
    T, Hd, V = shape
    inp = generate("medium", T=T, Hd=Hd, V=V)
    inp.targets[::7] = IGNORE_INDEX
    H, W, y, _ = to_device(inp, cuda_device)
    lib = flce.load_library()
    dev = cuda_device
    s = P(torch.cuda.current_stream(dev).cuda_stream)
    loss = Guarded((1,), torch.float32, dev)
    loss_rows = Guarded((T,), torch.float32, dev)
    lse = Guarded((T,), torch.float32, dev)
    logp = Guarded((T,), torch.float32, dev)
    nv = Guarded((1,), torch.int64, dev)
    fws = Guarded((lib.flce_forward_workspace_size(T, Hd, V),), torch.uint8, dev)
    assert lib.flce_forward(P(H.data_ptr()), P(W.data_ptr()), P(y.data_ptr()), T, Hd, V, IGNORE_INDEX, 1, _p(loss),
                            _p(lse), _p(logp), _p(nv), _p(fws), fws.nbytes, s) == 0
    assert lib.flce_forward(P(H.data_ptr()), P(W.data_ptr()), P(y.data_ptr()), T, Hd, V, IGNORE_INDEX, 0,
                            _p(loss_rows), _p(lse), _p(logp), _p(nv), _p(fws), fws.nbytes, s) == 0
    vws = Guarded((lib.flce_forward_valid_workspace_size(T, Hd, V),), torch.uint8, dev)
    vlse = Guarded((T,), torch.float32, dev)
    vlogp = Guarded((T,), torch.float32, dev)
    assert lib.flce_forward_valid(P(H.data_ptr()), P(W.data_ptr()), P(y.data_ptr()), T, Hd, V, IGNORE_INDEX, 0,
                                  _p(loss_rows), _p(vlse), _p(vlogp), _p(nv), _p(vws), vws.nbytes, s) == 0
    dloss = torch.ones(1, device=dev)
    dH = Guarded((T, Hd), torch.bfloat16, dev)
    dW = Guarded((V, Hd), torch.float32, dev)
    # a workspace for 128-token chunks: several chunks whenever T > 128
    bws_bytes = flce.flce_backward_workspace_size_for_chunk(T, Hd, V, 128)
    bws = Guarded((bws_bytes,), torch.uint8, dev)
    assert lib.flce_backward(P(dloss.data_ptr()), P(H.data_ptr()), P(W.data_ptr()), P(y.data_ptr()), _p(lse), T, Hd,
                             V, IGNORE_INDEX, 1, _p(dH), _p(dW), _p(bws), bws.nbytes, s) == 0
    sws = Guarded((lib.flce_score_workspace_size(T, Hd, V),), torch.uint8, dev)
    amax = Guarded((T,), torch.int64, dev)
    assert lib.flce_score(P(H.data_ptr()), P(W.data_ptr()), P(y.data_ptr()), T, Hd, V, IGNORE_INDEX, _p(logp),
                          _p(lse), _p(amax), _p(sws), sws.nbytes, s) == 0
    svws = Guarded((lib.flce_score_valid_workspace_size(T, Hd, V),), torch.uint8, dev)
    samax = Guarded((T,), torch.int64, dev)
    assert lib.flce_score_valid(P(H.data_ptr()), P(W.data_ptr()), P(y.data_ptr()), T, Hd, V, IGNORE_INDEX,
                                _p(vlogp), _p(vlse), _p(samax), _p(svws), svws.nbytes, s) == 0
    cut = max(1, V // 3)
    Wa = W[:cut].contiguous()
    slse = Guarded((T,), torch.float32, dev)
    szy = Guarded((T,), torch.float32, dev)
    assert lib.flce_forward_shard(P(H.data_ptr()), P(Wa.data_ptr()), P(y.data_ptr()), T, Hd, cut, 0, V, IGNORE_INDEX,
                                  _p(slse), _p(szy), _p(fws), fws.nbytes, s) == 0
    dHp = Guarded((T, Hd), torch.bfloat16, dev)
    dWs = Guarded((cut, Hd), torch.float32, dev)
    assert lib.flce_backward_shard(P(dloss.data_ptr()), P(H.data_ptr()), P(Wa.data_ptr()), P(y.data_ptr()), _p(lse),
                                   T, Hd, cut, 0, V, IGNORE_INDEX, 1, _p(dHp), _p(dWs), _p(bws), bws.nbytes, s) == 0
    torch.cuda.synchronize()
    for name, g in [("loss", loss), ("loss_rows", loss_rows), ("lse", lse), ("logp", logp), ("n_valid", nv),
                    ("fwd workspace", fws), ("dH", dH), ("dW", dW), ("bwd workspace", bws),
                    ("score workspace", sws), ("argmax", amax), ("shard_lse", slse), ("shard_zy", szy),
                    ("dH partial", dHp), ("dW shard", dWs), ("valid-forward workspace", vws),
                    ("valid-forward lse", vlse), ("valid-forward logp", vlogp),
                    ("valid-score workspace", svws), ("valid-score argmax", samax)]:
        assert g.intact(), name
    assert flce.flce_read_device_status(fws.t) == 0 and flce.flce_read_device_status(bws.t) == 0
