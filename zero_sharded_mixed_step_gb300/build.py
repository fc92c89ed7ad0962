"""Build libzero_gb300.so in-tree for sm_103a with nvcc (no CMake).

Translation units are compiled in parallel into ``_build/`` at the
repository root and linked into ``zero_sharded_mixed_step_gb300/libzero_gb300.so``
against the shared CUDA runtime (``libcudart.so``, found through the
library's run path in the toolkit), so that the library, PyTorch and a C
caller in one process share one runtime: device resets, errors and loaded
modules are seen alike by all of them.  Run
``python -m zero_sharded_mixed_step_gb300.build`` or call ``build()``.
"""

from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libzero_gb300.so")
SOURCES = ["zero_api.cpp", "host_step.cpp", "bucket_step.cpp", "fused_step.cu", "copy_cast.cu", "zero3_static.cu", "dp_replicas.cu",
           "host_memory.cpp", "offload_mean.cu", "offload.cpp"]
# Host arithmetic must match the device kernel's operation for operation: no
# contraction of a product and a sum into one fused operation by the compiler
# (the code writes every fused multiply-add it wants), and no errno from sqrt,
# which would keep the loop from being vectorised.
EXTRA_FLAGS = {"offload.cpp": ["-Xcompiler", "-ffp-contract=off", "-Xcompiler", "-fno-math-errno"]}
HEADERS = [os.path.join(CSRC, "zero_internal.h"), os.path.join(CSRC, "zero_context.h"), os.path.join(CSRC, "step_math.cuh"),
           os.path.join(INCLUDE, "zero_step.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    return os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"


def nvcc() -> str:
    path = os.path.join(cuda_home(), "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def cudart_dir() -> str:
    """The toolkit directory holding libcudart.so (the library's run path)."""
    home = cuda_home()
    for cand in [os.path.join(home, "lib64"), os.path.join(home, "lib")] + \
            sorted(glob.glob(os.path.join(home, "targets", "*", "lib"))):
        if os.path.exists(os.path.join(cand, "libcudart.so")):
            return cand
    return os.path.join(home, "lib64")


def _flags(ptxas_verbose: bool):
    f = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    return f


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd, verbose):
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"build step failed ({res.returncode}): {' '.join(cmd)}")
    return res


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile (only what changed, unless ``force``) and link; returns the library path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    objs, jobs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        if force or ptxas_verbose or _stale(obj, [path] + HEADERS):
            jobs.append([nvcc()] + _flags(ptxas_verbose) + EXTRA_FLAGS.get(src, []) + ["-c", path, "-o", obj])
    with ThreadPoolExecutor(max_workers=max(1, len(jobs))) as pool:
        list(pool.map(lambda c: _run(c, verbose or ptxas_verbose), jobs))
    if force or jobs or _stale(LIB, objs + [os.path.abspath(__file__)]):
        tmp = LIB + ".tmp"
        _run([nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-Xlinker", "-rpath", "-Xlinker", cudart_dir(),
                                 "-o", tmp] + objs, verbose)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_verbose="--ptxas" in sys.argv))
