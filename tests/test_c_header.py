"""include/flce.h is usable from plain C: a C99 program compiles against it with
warnings as errors, links the library and runs its host-only checks."""

import os
import shutil
import subprocess

import pytest

from lm_head_linear_gb300 import build as flce_build

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_header_compiles_as_c99_and_links(tmp_path):
    lib = flce_build.build()
    exe = tmp_path / "c_abi_host"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", flce_build.INCLUDE,
           os.path.join(HERE, "c_abi_host.c"), "-o", str(exe), "-L", os.path.dirname(lib), "-lflce",
           f"-Wl,-rpath,{os.path.dirname(lib)}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"
