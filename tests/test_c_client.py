"""The C ABI from plain C: the header compiles as C11, and (GPU) a C client
allocates with the CUDA runtime, runs a step and checks it."""

import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
SRC = os.path.join(HERE, "c_abi_client.c")


def _gcc(*extra):
    return ["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
            os.path.join(CUDA, "include"), SRC, *extra]


def test_header_and_client_compile_as_c11():
    res = subprocess.run(_gcc("-fsyntax-only"), capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


@pytest.mark.gpu
def test_c_client_runs_a_step(tmp_path):
    from zero_sharded_mixed_step_gb300 import build
    lib = build.build()
    exe = str(tmp_path / "c_client")
    libdir = os.path.dirname(lib)
    res = subprocess.run(_gcc("-o", exe, "-L", libdir, "-lzero_gb300", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                              "-lm", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"),
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "matches the closed form" in run.stdout
