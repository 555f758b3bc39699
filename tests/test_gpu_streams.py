"""Two independent problems on two CUDA streams at once, each with its own
workspaces: the library keeps no state between calls beyond the caller's
buffers, so both give bit-identical results to the same calls made one after
the other on one stream."""

import pytest
import torch

import lm_head_linear_gb300 as flce
from workloads import generate

from gpu_helpers import to_device

pytestmark = pytest.mark.gpu


def _problem(seed, dev):
    inp = generate("medium", T=2000, Hd=256, V=7000, seed=seed)
    return inp, to_device(inp, dev)


def _call(inp, tensors, stream):
    H, W, y, dl = tensors
    with torch.cuda.stream(stream):
        loss, lse, logp, nv, fws = flce.flce_forward(H, W, y, inp.ignore_index, inp.reduction, stream=stream)
        dH, dW, bws = flce.flce_backward(dl, H, W, y, lse, inp.ignore_index, inp.reduction, stream=stream)
    return {"loss": loss, "lse": lse, "logp": logp, "dH": dH, "dW": dW, "fws": fws, "bws": bws}


def test_two_streams_match_one_stream(cuda_device):
    a_inp, a = _problem(11, cuda_device)
    b_inp, b = _problem(12, cuda_device)
    s0 = torch.cuda.current_stream(cuda_device)
    seq = [_call(a_inp, a, s0), _call(b_inp, b, s0)]
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(cuda_device), torch.cuda.Stream(cuda_device)
    s1.wait_stream(s0)
    s2.wait_stream(s0)
    par = [_call(a_inp, a, s1), _call(b_inp, b, s2)]
    torch.cuda.synchronize()
    for x, y in zip(seq, par):
        for k in ("loss", "lse", "logp", "dH", "dW"):
            assert torch.equal(x[k], y[k]), k
        assert flce.flce_read_device_status(y["fws"]) == 0 and flce.flce_read_device_status(y["bws"]) == 0


def test_two_host_threads(cuda_device):
    """Two host threads call the library at the same time (ctypes releases the GIL during
    the calls), each on its own stream with its own buffers, five steps each: the results
    match the one-stream results bit for bit."""
    import threading

    probs = [_problem(21, cuda_device), _problem(22, cuda_device)]
    s0 = torch.cuda.current_stream(cuda_device)
    seq = [_call(inp, t, s0) for inp, t in probs]
    torch.cuda.synchronize()
    results, errors = [None, None], []

    def work(i):
        try:
            torch.cuda.set_device(cuda_device)
            st = torch.cuda.Stream(cuda_device)
            st.wait_stream(s0)
            for _ in range(5):
                results[i] = _call(probs[i][0], probs[i][1], st)
            st.synchronize()
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    assert not errors, errors
    torch.cuda.synchronize()
    for x, y in zip(seq, results):
        for k in ("loss", "lse", "logp", "dH", "dW"):
            assert torch.equal(x[k], y[k]), k
