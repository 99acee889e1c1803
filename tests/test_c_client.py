"""The C ABI from a C program (tests/c_client/step_tiny.c): no Python or
PyTorch between the caller and the library.

* CPU: include/dpg.h compiles as C11 with -Wall -Werror, and the client
  links against libdpg.so and the oracle.
* GPU: the client runs the tiny case (two steps and an all-gather) and
  matches the oracle bit for bit.
"""
import os
import subprocess

import pytest

import oracle
import zero_optimizer_step_gb300 as dpg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "step_tiny.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    from zero_optimizer_step_gb300 import build
    build.build()
    olib = oracle.build()
    exe = str(tmp_path / "step_tiny")
    libdir = os.path.dirname(dpg.LIB_PATH)
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", SRC, "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           dpg.LIB_PATH, olib, "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.dirname(olib)}",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_header_compiles_as_c_and_client_links(tmp_path):
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
def test_c_client_matches_oracle(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bit-exact" in r.stdout
