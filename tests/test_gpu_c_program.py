"""The C ABI from a plain C program on the GPU: the program allocates device
memory itself (cudaMalloc), runs flce_forward and flce_backward, and its
outputs match the fp64 oracle."""

import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from lm_head_linear_gb300 import build as flce_build
from workloads import bf16_bits_to_f64, generate

from gpu_helpers import TOL_GRAD, TOL_TOKEN, rel_fro

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_program_forward_backward(tmp_path, cuda_device):
    lib = flce_build.build()
    exe = tmp_path / "c_abi_gpu"
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-I", flce_build.INCLUDE, "-I", os.path.join(CUDA, "include"),
           os.path.join(HERE, "c_abi_gpu.c"), "-o", str(exe), "-L", os.path.dirname(lib), "-lflce",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.dirname(lib)}",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    T, Hd, V = 500, 192, 3001
    inp = generate("medium", T=T, Hd=Hd, V=V)
    inp.H_bits.tofile(tmp_path / "H.bin")
    inp.W_bits.tofile(tmp_path / "W.bin")
    inp.targets.astype(np.int64).tofile(tmp_path / "y.bin")
    r = subprocess.run([str(exe), str(tmp_path), str(T), str(Hd), str(V)], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    lse = np.fromfile(tmp_path / "lse.bin", dtype=np.float32)
    logp = np.fromfile(tmp_path / "logp.bin", dtype=np.float32)
    loss = np.fromfile(tmp_path / "loss.bin", dtype=np.float32)[0]
    dH = bf16_bits_to_f64(np.fromfile(tmp_path / "dH.bin", dtype=np.uint16).reshape(T, Hd))
    dW = np.fromfile(tmp_path / "dW.bin", dtype=np.float32).reshape(V, Hd)
    ref = oracle.forward(inp.H64(), inp.W64(), inp.targets, inp.ignore_index, "mean")
    assert np.max(np.abs(lse - ref.lse)) <= TOL_TOKEN
    assert np.max(np.abs(logp - ref.logp)) <= TOL_TOKEN
    assert abs(float(loss) - float(ref.loss)) <= TOL_TOKEN
    dH_ref, dW_ref = oracle.backward(1.0, inp.H64(), inp.W64(), inp.targets, inp.ignore_index, "mean")
    assert rel_fro(dH, dH_ref) <= TOL_GRAD
    assert rel_fro(dW, dW_ref) <= TOL_GRAD
