"""ctypes binding of ``libflce.so`` (the C ABI in ``include/flce.h``).

Argument marshalling only: tensors are checked, output / workspace buffers are
allocated with torch (device-memory plumbing), and every step of the
computation runs in the library's CUDA kernels.  There is no CPU or PyTorch
fallback: if the library is missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

# Where `python -m lm_head_linear_gb300.build` writes the library.
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libflce.so")

REDUCTIONS = {"none": 0, "mean": 1, "sum": 2}
STATUS_NAMES = {
    0: "FLCE_OK", 1: "FLCE_ERR_INVALID_ARG", 2: "FLCE_ERR_UNSUPPORTED", 3: "FLCE_ERR_ALIGNMENT",
    4: "FLCE_ERR_WORKSPACE", 5: "FLCE_ERR_CUDA", 6: "FLCE_ERR_TARGET_RANGE", 7: "FLCE_ERR_TIMEOUT",
}
KERNEL_KINDS = 9
ABI_VERSION = 2  # FLCE_ABI_VERSION of include/flce.h

# Every symbol the header declares: name -> (restype, argtypes).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
SIGNATURES = {
    "flce_forward_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64]),
    "flce_backward_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64]),
    "flce_forward_valid_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64]),
    "flce_backward_workspace_size_for_chunk": (ctypes.c_size_t, [_I64, _I64, _I64, _I64]),
    "flce_backward_chunk_tokens": (_I64, [_I64, _I64, _I64, ctypes.c_size_t]),
    "flce_forward": (_I32, [_P, _P, _P, _I64, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "flce_forward_valid": (_I32, [_P, _P, _P, _I64, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "flce_forward_noalloc": (_I32, [_P, _P, _P, _I64, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, _P]),
    "flce_score_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64]),
    "flce_score_valid_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64]),
    "flce_score": (_I32, [_P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "flce_score_valid": (_I32, [_P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "flce_forward_shard": (_I32, [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, ctypes.c_size_t, _P]),
    "flce_combine_workspace_size": (ctypes.c_size_t, [_I64, _I32]),
    "flce_combine_shards": (_I32, [_P, _P, _I32, _P, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                   _P]),
    "flce_backward_shard": (_I32, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I32, _P, _P, _P,
                                   ctypes.c_size_t, _P]),
    "flce_backward": (_I32, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I32, _P, _P, _P, ctypes.c_size_t, _P]),
    "flce_backward_logp": (_I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I32, _P, _P, _P, ctypes.c_size_t,
                                  _P]),
    "flce_read_device_status": (_I32, [_P, _P, ctypes.POINTER(_I32)]),
    "flce_selftest_wait_timeout": (_I32, [_P, ctypes.c_uint64, _P]),
    "flce_status_string": (ctypes.c_char_p, [_I32]),
    "flce_last_error": (ctypes.c_char_p, []),
    "flce_abi_version": (_I32, []),
    "flce_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "flce_profile_enable": (None, [_I32]),
    "flce_profile_collect": (_I32, [_P, _I32, ctypes.POINTER(_I32)]),
    "flce_kernel_name": (ctypes.c_char_p, [_I32]),
}


class KernelStats(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


class FlceError(RuntimeError):
    def __init__(self, status: int, detail: str = ""):
        self.status = int(status)
        super().__init__(f"{STATUS_NAMES.get(self.status, self.status)}: {detail}")


_LIB: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load the in-tree library (raises if it was not built)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -m lm_head_linear_gb300.build` "
                               "(there is no fallback implementation)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if lib.flce_abi_version() != ABI_VERSION:
            raise RuntimeError(f"libflce ABI version {lib.flce_abi_version()}, this binding needs {ABI_VERSION}")
        _LIB = lib
    return _LIB


def _check(status: int):
    if status != 0:
        lib = load_library()
        raise FlceError(status, (lib.flce_last_error() or b"").decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_inputs(H: torch.Tensor, W: torch.Tensor, targets: torch.Tensor):
    if not (H.is_cuda and W.is_cuda and targets.is_cuda):
        raise ValueError("H, W and targets must be CUDA tensors")
    if H.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise ValueError("H and W must be bfloat16")
    if targets.dtype != torch.int64:
        raise ValueError("targets must be int64")
    if H.dim() != 2 or W.dim() != 2 or targets.dim() != 1:
        raise ValueError("H [T, Hd], W [V, Hd], targets [T]")
    if H.shape[1] != W.shape[1] or H.shape[0] != targets.shape[0]:
        raise ValueError(f"shape mismatch: H {tuple(H.shape)}, W {tuple(W.shape)}, targets {tuple(targets.shape)}")
    if not (H.is_contiguous() and W.is_contiguous() and targets.is_contiguous()):
        raise ValueError("H, W and targets must be contiguous")
    if not (H.device == W.device == targets.device):
        raise ValueError("H, W and targets must be on one device")


def _check_rows(name: str, t: torch.Tensor, shape, dtype, device):
    """A device array the library reads through its pointer: same device, dtype, shape."""
    if t.device != device or t.dtype != dtype or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be a {dtype} tensor of shape {tuple(shape)} on {device}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")


def flce_forward_workspace_size(T: int, Hd: int, V: int) -> int:
    return int(load_library().flce_forward_workspace_size(T, Hd, V))


def flce_backward_workspace_size(T: int, Hd: int, V: int) -> int:
    return int(load_library().flce_backward_workspace_size(T, Hd, V))


def flce_backward_workspace_size_for_chunk(T: int, Hd: int, V: int, chunk: int) -> int:
    return int(load_library().flce_backward_workspace_size_for_chunk(T, Hd, V, chunk))


def flce_backward_chunk_tokens(T: int, Hd: int, V: int, workspace_bytes: int) -> int:
    return int(load_library().flce_backward_chunk_tokens(T, Hd, V, workspace_bytes))


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if workspace.device != device or workspace.dtype != torch.uint8 or not workspace.is_contiguous():
        raise ValueError(f"the workspace must be a contiguous uint8 tensor on {device}")
    return workspace


def _out(out: Optional[dict], key: str, shape, dtype, device) -> torch.Tensor:
    """out[key] if the caller gave one (checked: the library writes through its pointer),
    else a new tensor."""
    t = (out or {}).get(key)
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    want = (shape,) if isinstance(shape, int) else tuple(shape)
    if tuple(t.shape) != want or t.dtype != dtype or t.device != device or not t.is_contiguous():
        raise ValueError(f"out[{key!r}] must be a contiguous {dtype} tensor of shape {want} on {device}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")
    return t


def flce_forward(H: torch.Tensor, W: torch.Tensor, targets: torch.Tensor, ignore_index: int = -100,
                 reduction: str = "mean", workspace: Optional[torch.Tensor] = None, stream=None,
                 out: Optional[dict] = None):
    """Run ``flce_forward``; returns ``(loss, lse, logp, n_valid, workspace)``.

    ``loss`` is a 1-element fp32 tensor (mean / sum) or [T] (none); ``n_valid``
    a 1-element int64 tensor.  ``out`` may hold preallocated ``loss``, ``lse``,
    ``logp`` and ``n_valid`` tensors.
    """
    return _forward("flce_forward", "flce_forward_workspace_size", H, W, targets, ignore_index, reduction,
                    workspace, stream, out)


def flce_forward_valid(H: torch.Tensor, W: torch.Tensor, targets: torch.Tensor, ignore_index: int = -100,
                       reduction: str = "mean", workspace: Optional[torch.Tensor] = None, stream=None,
                       out: Optional[dict] = None):
    """Run ``flce_forward_valid``: as :func:`flce_forward`, but rows with an ignored
    target are not computed (their lse is 0).  Same return values."""
    return _forward("flce_forward_valid", "flce_forward_valid_workspace_size", H, W, targets, ignore_index,
                    reduction, workspace, stream, out)


def flce_forward_valid_workspace_size(T: int, Hd: int, V: int) -> int:
    return int(load_library().flce_forward_valid_workspace_size(T, Hd, V))


def _forward(entry, size_fn, H, W, targets, ignore_index, reduction, workspace, stream, out):
    _check_inputs(H, W, targets)
    lib = load_library()
    T, Hd = H.shape
    V = W.shape[0]
    red = REDUCTIONS[reduction]
    dev = H.device
    loss = _out(out, "loss", T if red == 0 else 1, torch.float32, dev)
    lse = _out(out, "lse", T, torch.float32, dev)
    logp = _out(out, "logp", T, torch.float32, dev)
    n_valid = _out(out, "n_valid", 1, torch.int64, dev)
    need = getattr(lib, size_fn)(T, Hd, V)
    ws = _workspace(need, dev, workspace)
    st = getattr(lib, entry)(_ptr(H), _ptr(W), _ptr(targets), T, Hd, V, int(ignore_index), red, _ptr(loss),
                             _ptr(lse), _ptr(logp), _ptr(n_valid), _ptr(ws), ws.numel(), _stream_handle(stream))
    _check(st)
    return loss, lse, logp, n_valid, ws


def flce_backward(dloss: Optional[torch.Tensor], H: torch.Tensor, W: torch.Tensor, targets: torch.Tensor,
                  lse: torch.Tensor, ignore_index: int = -100, reduction: str = "mean",
                  workspace: Optional[torch.Tensor] = None, stream=None, out: Optional[dict] = None,
                  dlogp: Optional[torch.Tensor] = None):
    """Run ``flce_backward`` (or ``flce_backward_logp`` when ``dlogp``, a [T] gradient on
    the logp output, is given; ``dloss`` may then be None).  Returns
    ``(dH bf16 [T, Hd], dW fp32 [V, Hd], workspace)``."""
    _check_inputs(H, W, targets)
    lib = load_library()
    T, Hd = H.shape
    V = W.shape[0]
    red = REDUCTIONS[reduction]
    dev = H.device
    if dloss is None and dlogp is None:
        raise ValueError("give dloss, dlogp or both")
    if dloss is not None:
        dloss = dloss.to(device=dev, dtype=torch.float32).contiguous().reshape(-1)
        if dloss.numel() != (T if red == 0 else 1):
            raise ValueError("dloss must have one element (mean / sum) or T elements (none)")
    if dlogp is not None:
        dlogp = dlogp.to(device=dev, dtype=torch.float32).contiguous().reshape(-1)
        if dlogp.numel() != T:
            raise ValueError("dlogp must have T elements")
    _check_rows("lse", lse, (T,), torch.float32, dev)
    lse = lse.contiguous()
    dH = _out(out, "dH", (T, Hd), torch.bfloat16, dev)
    dW = _out(out, "dW", (V, Hd), torch.float32, dev)
    need = lib.flce_backward_workspace_size(T, Hd, V)
    ws = _workspace(need, dev, workspace)
    if dlogp is None:
        st = lib.flce_backward(_ptr(dloss), _ptr(H), _ptr(W), _ptr(targets), _ptr(lse), T, Hd, V, int(ignore_index),
                               red, _ptr(dH), _ptr(dW), _ptr(ws), ws.numel(), _stream_handle(stream))
    else:
        st = lib.flce_backward_logp(_ptr(dloss), _ptr(dlogp), _ptr(H), _ptr(W), _ptr(targets), _ptr(lse), T, Hd, V,
                                    int(ignore_index), red, _ptr(dH), _ptr(dW), _ptr(ws), ws.numel(),
                                    _stream_handle(stream))
    _check(st)
    return dH, dW, ws




def flce_score(H: torch.Tensor, W: torch.Tensor, targets: torch.Tensor, ignore_index: int = -100,
               workspace: Optional[torch.Tensor] = None, stream=None, out: Optional[dict] = None):
    """Run ``flce_score``; returns ``(logp [T] fp32, lse [T] fp32, argmax [T] int64, workspace)``.
    ``out`` may hold preallocated ``logp``, ``lse`` and ``argmax`` tensors."""
    return _score("flce_score", "flce_score_workspace_size", H, W, targets, ignore_index, workspace, stream, out)


def flce_score_valid(H: torch.Tensor, W: torch.Tensor, targets: torch.Tensor, ignore_index: int = -100,
                     workspace: Optional[torch.Tensor] = None, stream=None, out: Optional[dict] = None):
    """Run ``flce_score_valid``: as :func:`flce_score` on the rows with a valid target;
    rows with an ignored target are not computed (lse 0, logp 0, argmax -1)."""
    return _score("flce_score_valid", "flce_score_valid_workspace_size", H, W, targets, ignore_index, workspace,
                  stream, out)


def _score(entry, size_fn, H, W, targets, ignore_index, workspace, stream, out):
    _check_inputs(H, W, targets)
    lib = load_library()
    T, Hd = H.shape
    V = W.shape[0]
    dev = H.device
    logp = _out(out, "logp", T, torch.float32, dev)
    lse = _out(out, "lse", T, torch.float32, dev)
    argmax = _out(out, "argmax", T, torch.int64, dev)
    ws = _workspace(getattr(lib, size_fn)(T, Hd, V), dev, workspace)
    _check(getattr(lib, entry)(_ptr(H), _ptr(W), _ptr(targets), T, Hd, V, int(ignore_index), _ptr(logp), _ptr(lse),
                               _ptr(argmax), _ptr(ws), ws.numel(), _stream_handle(stream)))
    return logp, lse, argmax, ws


def flce_forward_shard(H: torch.Tensor, W_shard: torch.Tensor, targets: torch.Tensor, vocab_offset: int,
                       V_total: int, ignore_index: int = -100, workspace: Optional[torch.Tensor] = None, stream=None,
                       out: Optional[dict] = None):
    """Run ``flce_forward_shard``; returns ``(shard_lse [T], shard_zy [T], workspace)``.
    ``out`` may hold preallocated ``shard_lse`` and ``shard_zy`` tensors."""
    _check_inputs(H, W_shard, targets)
    lib = load_library()
    T, Hd = H.shape
    Vs = W_shard.shape[0]
    dev = H.device
    shard_lse = _out(out, "shard_lse", T, torch.float32, dev)
    shard_zy = _out(out, "shard_zy", T, torch.float32, dev)
    ws = _workspace(lib.flce_forward_workspace_size(T, Hd, Vs), dev, workspace)
    _check(lib.flce_forward_shard(_ptr(H), _ptr(W_shard), _ptr(targets), T, Hd, Vs, int(vocab_offset), int(V_total),
                                  int(ignore_index), _ptr(shard_lse), _ptr(shard_zy), _ptr(ws), ws.numel(),
                                  _stream_handle(stream)))
    return shard_lse, shard_zy, ws


def flce_combine_shards(shard_lse: torch.Tensor, shard_zy: torch.Tensor, targets: torch.Tensor, V_total: int,
                        ignore_index: int = -100, reduction: str = "mean", workspace: Optional[torch.Tensor] = None,
                        stream=None, out: Optional[dict] = None):
    """Run ``flce_combine_shards`` on [n_shards, T] partials; returns ``(loss, lse, logp, n_valid, workspace)``.
    ``out`` may hold preallocated ``loss``, ``lse``, ``logp`` and ``n_valid`` tensors."""
    lib = load_library()
    if shard_lse.dim() != 2 or not shard_lse.is_cuda:
        raise ValueError("shard_lse must be a CUDA tensor [n_shards, T]")
    n_shards, T = shard_lse.shape
    dev = shard_lse.device
    _check_rows("shard_lse", shard_lse, (n_shards, T), torch.float32, dev)
    _check_rows("shard_zy", shard_zy, (n_shards, T), torch.float32, dev)
    _check_rows("targets", targets, (T,), torch.int64, dev)
    shard_lse = shard_lse.contiguous()
    shard_zy = shard_zy.contiguous()
    targets = targets.contiguous()
    red = REDUCTIONS[reduction]
    loss = _out(out, "loss", T if red == 0 else 1, torch.float32, dev)
    lse = _out(out, "lse", T, torch.float32, dev)
    logp = _out(out, "logp", T, torch.float32, dev)
    n_valid = _out(out, "n_valid", 1, torch.int64, dev)
    ws = _workspace(lib.flce_combine_workspace_size(T, n_shards), dev, workspace)
    _check(lib.flce_combine_shards(_ptr(shard_lse), _ptr(shard_zy), n_shards, _ptr(targets), T, int(V_total),
                                   int(ignore_index), red, _ptr(loss), _ptr(lse), _ptr(logp), _ptr(n_valid),
                                   _ptr(ws), ws.numel(), _stream_handle(stream)))
    return loss, lse, logp, n_valid, ws


def flce_backward_shard(dloss: torch.Tensor, H: torch.Tensor, W_shard: torch.Tensor, targets: torch.Tensor,
                        lse: torch.Tensor, vocab_offset: int, V_total: int, ignore_index: int = -100,
                        reduction: str = "mean", workspace: Optional[torch.Tensor] = None, stream=None,
                        out: Optional[dict] = None):
    """Run ``flce_backward_shard``; returns ``(dH_partial bf16 [T, Hd], dW_shard fp32 [V_shard, Hd], workspace)``.
    ``out`` may hold preallocated ``dH`` and ``dW`` tensors."""
    _check_inputs(H, W_shard, targets)
    lib = load_library()
    T, Hd = H.shape
    Vs = W_shard.shape[0]
    red = REDUCTIONS[reduction]
    dev = H.device
    dloss = dloss.to(device=dev, dtype=torch.float32).contiguous().reshape(-1)
    if dloss.numel() != (T if red == 0 else 1):
        raise ValueError("dloss must have one element (mean / sum) or T elements (none)")
    _check_rows("lse", lse, (T,), torch.float32, dev)
    dH = _out(out, "dH", (T, Hd), torch.bfloat16, dev)
    dW = _out(out, "dW", (Vs, Hd), torch.float32, dev)
    ws = _workspace(lib.flce_backward_workspace_size(T, Hd, Vs), dev, workspace)
    _check(lib.flce_backward_shard(_ptr(dloss), _ptr(H), _ptr(W_shard), _ptr(targets), _ptr(lse.contiguous()), T, Hd,
                                   Vs, int(vocab_offset), int(V_total), int(ignore_index), red, _ptr(dH), _ptr(dW),
                                   _ptr(ws), ws.numel(), _stream_handle(stream)))
    return dH, dW, ws


def flce_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    lib = load_library()
    v = ctypes.c_int32(-1)
    _check(lib.flce_read_device_status(_ptr(workspace), _stream_handle(stream), ctypes.byref(v)))
    return int(v.value)


def flce_selftest_wait_timeout(timeout_ns: int, device=None, stream=None) -> int:
    """Run the bounded-wait self-test; returns the device status it produced."""
    lib = load_library()
    ws = torch.empty(256, dtype=torch.uint8, device=device or torch.device("cuda"))
    _check(lib.flce_selftest_wait_timeout(_ptr(ws), int(timeout_ns), _stream_handle(stream)))
    return flce_read_device_status(ws, stream)


def flce_set_wait_timeout_ns(ns: int):
    load_library().flce_set_wait_timeout_ns(int(ns))


def flce_profile_enable(on: bool = True):
    load_library().flce_profile_enable(1 if on else 0)


def flce_profile_collect() -> dict:
    """Per-kernel-kind {name: {launches, total_ms, flops, bytes}} since the last collect."""
    lib = load_library()
    arr = (KernelStats * KERNEL_KINDS)()
    n = ctypes.c_int32(0)
    _check(lib.flce_profile_collect(ctypes.cast(arr, ctypes.c_void_p), KERNEL_KINDS, ctypes.byref(n)))
    res = {}
    for i in range(n.value):
        r = arr[i]
        res[lib.flce_kernel_name(r.kind).decode()] = {
            "launches": int(r.launches), "total_ms": float(r.total_ms), "flops": float(r.flops),
            "bytes": float(r.bytes)}
    return res


class LinearCrossEntropy(torch.autograd.Function):
    """autograd wrapper: forward runs ``flce_forward_valid`` (rows with an ignored target
    cost nothing), backward ``flce_backward`` (``flce_backward_logp`` when a gradient
    reaches ``logp``).

    Returns ``(loss, logp)``; both are differentiable, so an objective built
    from the per-token log-probabilities (e.g. ``-(adv * logp).sum()``) works.
    The weight gradient comes back in W's dtype.
    """

    @staticmethod
    def forward(ctx, H, W, targets, ignore_index: int = -100, reduction: str = "mean"):
        loss, lse, logp, _, _ = flce_forward_valid(H, W, targets, ignore_index, reduction)
        ctx.save_for_backward(H, W, targets, lse)
        ctx.ignore_index = ignore_index
        ctx.reduction = reduction
        if reduction != "none":
            loss = loss.reshape(())
        return loss, logp

    @staticmethod
    def backward(ctx, dloss, dlogp):
        H, W, targets, lse = ctx.saved_tensors
        dH, dW, _ = flce_backward(dloss, H, W, targets, lse, ctx.ignore_index, ctx.reduction, dlogp=dlogp)
        return dH, dW.to(W.dtype), None, None, None


def linear_cross_entropy(H, W, targets, ignore_index: int = -100, reduction: str = "mean"):
    """Fused ``cross_entropy(H @ W.T, targets)`` without materialising the logits; returns the loss."""
    return LinearCrossEntropy.apply(H, W, targets, ignore_index, reduction)[0]


def linear_log_probs(H, W, targets, ignore_index: int = -100):
    """Per-token ``log p(target)`` under ``softmax(H @ W.T)`` (0 on ignored rows),
    differentiable, without materialising the logits."""
    return LinearCrossEntropy.apply(H, W, targets, ignore_index, "none")[1]
