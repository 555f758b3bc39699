"""The C-ABI library builds, loads, and exports every symbol include/flce.h declares.

No compute call is made here (no GPU needed); host-only entry points
(workspace sizing, status strings, ABI version, argument checks) are exercised.
"""

import ctypes
import os
import re
import subprocess

import pytest

import lm_head_linear_gb300 as flce
from lm_head_linear_gb300 import build as flce_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flce.h")


def declared_symbols():
    src = open(HEADER, encoding="utf-8").read()
    return sorted(set(re.findall(r"FLCE_API\s+[\w\s\*]+?\b(flce_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    flce_build.build()
    return flce.load_library()


def test_header_declares_the_two_calls():
    syms = declared_symbols()
    assert "flce_forward" in syms and "flce_backward" in syms
    assert len(syms) >= 13


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in flce.SIGNATURES, f"binding lacks a signature for {name}"


def test_exported_symbols_are_only_the_declared_ones(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", flce_build.LIB_PATH], capture_output=True, text=True).stdout
    exported = sorted({ln.split()[-1] for ln in out.splitlines()
                       if " T " in ln and ln.split()[-1].startswith("flce_")})
    assert exported == declared_symbols()


def test_host_only_entry_points(lib):
    assert lib.flce_abi_version() == 2
    assert lib.flce_status_string(0) == b"FLCE_OK"
    assert lib.flce_status_string(6) == b"FLCE_ERR_TARGET_RANGE"
    assert lib.flce_kernel_name(4) == b"bwd_dz"
    T, Hd, V = 65536, 2048, 124160
    fws = lib.flce_forward_workspace_size(T, Hd, V)
    bws = lib.flce_backward_workspace_size(T, Hd, V)
    assert 0 < fws < 64 * 2**20
    # the backward keeps a [chunk x V] bf16 slice of dZ, never [T x V]
    assert bws < T * V * 2
    chunk = lib.flce_backward_chunk_tokens(T, Hd, V, bws)
    assert 128 <= chunk < T and chunk % 128 == 0
    assert bws >= chunk * V * 2
    assert lib.flce_backward_chunk_tokens(T, Hd, V, 1024) == 0
    # a bigger workspace gives a bigger chunk, capped at T rounded up to 128
    assert lib.flce_backward_chunk_tokens(T, Hd, V, bws * 4) > chunk
    assert lib.flce_backward_chunk_tokens(1000, 64, 50, 2**30) == 1024
    for t in (257, 1000, 8192, 131072):
        assert lib.flce_backward_workspace_size(t, 4096, 124160) < t * 124160 * 2


def test_argument_errors_return_before_any_launch(lib):
    # Host-side validation needs no device: bad sizes and NULLs are rejected first.
    P = ctypes.c_void_p
    st = lib.flce_forward(P(16), P(16), P(16), 10, 100, 50, -100, 1, P(16), P(16), P(16), None, P(256), 1 << 20, None)
    assert st == 2  # Hd not a multiple of 64
    st = lib.flce_forward(P(16), P(16), P(16), 10, 64, 50, 3, 1, P(16), P(16), P(16), None, P(256), 1 << 20, None)
    assert st == 1  # ignore_index inside [0, V)
    st = lib.flce_forward(P(16), P(16), P(16), 10, 64, 50, -100, 7, P(16), P(16), P(16), None, P(256), 1 << 20, None)
    assert st == 1  # unknown reduction
    st = lib.flce_forward(P(16), P(18), P(16), 10, 64, 50, -100, 1, P(16), P(16), P(16), None, P(256), 1 << 20, None)
    assert st == 3  # misaligned W
    st = lib.flce_forward(P(16), P(16), P(16), 10, 64, 50, -100, 1, P(16), P(16), P(16), None, P(256), 16, None)
    assert st == 4  # workspace too small
    st = lib.flce_backward(P(16), P(16), P(16), P(16), P(16), 10, 64, 50, -100, 1, P(16), P(16), P(256), 16, None)
    assert st == 4
    st = lib.flce_forward(None, P(16), P(16), 10, 64, 50, -100, 1, P(16), P(16), P(16), None, P(256), 1 << 20, None)
    assert st == 1
    assert b"NULL" in lib.flce_last_error()


def test_misaligned_typed_arrays_are_rejected_on_the_host(lib):
    """Per-token arrays are accessed with typed loads and stores: a pointer off its
    element alignment is an argument error, returned before anything is launched."""
    P = ctypes.c_void_p
    ok = dict(H=P(16), W=P(16), y=P(16), loss=P(16), lse=P(16), logp=P(16), nv=P(16))

    def fwd(**kw):
        a = {**ok, **kw}
        return lib.flce_forward(a["H"], a["W"], a["y"], 10, 64, 50, -100, 1, a["loss"], a["lse"], a["logp"], a["nv"],
                                P(256), 1 << 20, None)

    assert fwd(y=P(20)) == 3       # targets (int64) off by 4
    assert fwd(lse=P(18)) == 3     # float off by 2
    assert fwd(logp=P(17)) == 3
    assert fwd(loss=P(19)) == 3
    assert fwd(nv=P(20)) == 3      # n_valid (int64) off by 4
    st = lib.flce_backward(P(18), P(16), P(16), P(16), P(16), 10, 64, 50, -100, 1, P(16), P(16), P(256), 1 << 30,
                           None)
    assert st == 3                 # dloss off by 2
    st = lib.flce_backward(P(16), P(16), P(16), P(16), P(22), 10, 64, 50, -100, 1, P(16), P(16), P(256), 1 << 30,
                           None)
    assert st == 3                 # lse off by 2
    st = lib.flce_score(P(16), P(16), P(16), 10, 64, 50, -100, P(16), P(16), P(12), P(256), 1 << 30, None)
    assert st == 3                 # argmax (int64) off by 4
    st = lib.flce_combine_shards(P(16), P(18), 2, P(16), 10, 50, -100, 1, P(16), P(16), P(16), P(16), P(256), 1 << 20,
                                 None)
    assert st == 3                 # shard_zy off by 2
    st = lib.flce_forward_shard(P(16), P(16), P(16), 10, 64, 25, 0, 50, -100, P(16), P(14), P(256), 1 << 20, None)
    assert st == 3


def test_noalloc_forward_size_limit_on_the_host(lib):
    """flce_forward_noalloc's built-in scratch holds 32 MiB: the documented maximum of
    253,952 tokens fits it at any Hd and V, one 128-token step more does not.  At the
    maximum the size check passes and the next argument check (a NULL H) answers; above
    it the call is refused as a workspace error.  Nothing is launched either way."""
    for Hd in (64, 2048, 4096, 16384):
        for V in (1, 4096, 124160, 300001):
            assert lib.flce_forward_workspace_size(253952, Hd, V) <= 32 << 20
            assert lib.flce_forward_workspace_size(253952 + 128, Hd, V) > 32 << 20
    P = ctypes.c_void_p
    st = lib.flce_forward_noalloc(None, P(16), P(16), 253952, 64, 300, -100, 1, P(16), P(16), P(16), None, None,
                                  None)
    assert st == 1 and b"NULL" in lib.flce_last_error()
    st = lib.flce_forward_noalloc(P(16), P(16), P(16), 253952 + 128, 64, 300, -100, 1, P(16), P(16), P(16), None,
                                  None, None)
    assert st == 4 and b"scratch" in lib.flce_last_error()


def test_backward_workspace_for_a_chunk_round_trips(lib):
    """flce_backward_workspace_size_for_chunk(c) is the smallest workspace that runs
    chunks of c rows (capped at T rounded up to 128), on ragged and large shapes."""
    for T, Hd, V in [(1, 64, 1), (300, 64, 4097), (8192, 2048, 124160), (65536, 4096, 248320)]:
        cap = -(-T // 128) * 128
        for c in (128, 256, 4096, 8192, 16384):
            w = lib.flce_backward_workspace_size_for_chunk(T, Hd, V, c)
            assert lib.flce_backward_chunk_tokens(T, Hd, V, w) == min(c, cap)
            assert lib.flce_backward_chunk_tokens(T, Hd, V, w - 1) < min(c, cap)
        default = cap if T <= 256 else min(8192, max(128, T // 2 // 128 * 128))
        assert lib.flce_backward_chunk_tokens(T, Hd, V, lib.flce_backward_workspace_size(T, Hd, V)) == default
    assert lib.flce_backward_workspace_size_for_chunk(1000, 64, 50, 100) == 0   # not a multiple of 128
    assert lib.flce_backward_workspace_size_for_chunk(1000, 64, 50, 0) == 0


def test_size_limits_are_argument_errors(lib):
    """T and V must stay below 2^30 (tile coordinates stay in int32), Hd below 2^24."""
    P = ctypes.c_void_p
    args = lambda T, Hd, V: (P(16), P(16), P(16), T, Hd, V, -100, 1, P(16), P(16), P(16), None, P(256), 1 << 40, None)
    assert lib.flce_forward(*args(1 << 30, 64, 50)) == 1
    assert lib.flce_forward(*args(10, 64, 1 << 30)) == 1
    assert lib.flce_forward(*args(10, 1 << 24, 50)) == 1
    assert lib.flce_forward(*args(-1, 64, 50)) == 1
    assert lib.flce_forward(*args(10, 64, 0)) == 1
    assert lib.flce_forward_valid(*args(1 << 30, 64, 50)) == 1
    assert lib.flce_backward_workspace_size(-1, 64, 50) == 0
    assert lib.flce_forward_workspace_size(10, 64, 0) == 0


def test_binding_and_header_agree_on_the_abi_version():
    import re

    import lm_head_linear_gb300.binding as b
    with open(os.path.join(ROOT, "include", "flce.h")) as fh:
        m = re.search(r"#define FLCE_ABI_VERSION (\d+)", fh.read())
    assert m and int(m.group(1)) == b.ABI_VERSION
