"""Compile the CUDA library in-tree for GB300 (sm_103a) with nvcc.

The shared library ``libmla_decode.so`` lands next to this file.  Host code
is portable C++ (no architecture-specific intrinsics), so the same sources
build on x86_64 and aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB_PATH = os.path.join(HERE, "libmla_decode.so")
SOURCES = ["api.cu", "plan.cpp", "prologue.cu"]
GENCODE = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def needs_build(out: str = LIB_PATH) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "mla_decode.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(out: str = LIB_PATH, verbose: bool = False, extra=()) -> str:
    cmd = [nvcc(), GENCODE, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
           f"-I{INCLUDE}", *extra, *[os.path.join(CSRC, s) for s in SOURCES], "-o", out]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    return out


if __name__ == "__main__":
    build(verbose=True)
    print(LIB_PATH)
