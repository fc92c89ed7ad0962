"""The one-launch forward gather of a ZeRO-3 step, checked directly from C++
(tests/cpp_gather_units.cpp): in a whole step the backward pass overwrites
both unit buffers, so the forward gathers' result is checked here, bit for
bit, with guard bytes around the buffers."""

import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_gather_units_leaves_each_buffer_holding_the_last_unit_of_its_parity(tmp_path):
    from zero_sharded_mixed_step_gb300 import build
    lib = build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "cpp_gather_units")
    res = subprocess.run(["g++", "-std=c++17", "-Wall", "-Werror", "-I", os.path.join(libdir, "csrc"), "-I",
                          os.path.join(ROOT, "include"), "-I", os.path.join(build.cuda_home(), "include"),
                          os.path.join(HERE, "cpp_gather_units.cpp"), "-o", exe, "-L", libdir, "-lzero_gb300",
                          "-L", build.cudart_dir(), "-lcudart", f"-Wl,-rpath,{libdir}",
                          f"-Wl,-rpath,{build.cudart_dir()}"], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "every buffer position holds the last unit of its parity" in run.stdout
