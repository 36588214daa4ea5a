"""Build libfp8fg.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

    python -m fp8_fine_grained_22_b300.build [--force]

IEEE semantics are kept on purpose: no --use_fast_math, no flush-to-zero,
no approximate division (the quantiser's codes must be exact functions of
their inputs).
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB_PATH = os.path.join(HERE, "libfp8fg.so")
SOURCES = [os.path.join(CSRC, f) for f in ("quant.cu", "gemm.cu", "dispatch.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("ptx.cuh", "common.cuh", "tensormap.cuh", "quant_math.cuh")] + [
    os.path.join(INCLUDE, "fp8fg.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared", "-ftz=false", "-prec-div=true",
              "-prec-sqrt=true", "-fmad=true"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    tmp = LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = [nvcc(), *NVCC_FLAGS, "-I", INCLUDE, *SOURCES, "-o", tmp]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
