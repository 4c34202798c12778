"""Build libssm_b300.so in-tree with nvcc for sm_103a (B300).

    python -m selective_state_space_137_b300.build
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libssm_b300.so")
SOURCES = [os.path.join(PKG, "csrc", "ssm_api.cu")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _deps():
    return SOURCES + glob.glob(os.path.join(PKG, "csrc", "*.cuh")) + \
        [os.path.join(ROOT, "include", "ssm.h")]


def nvcc_command(out: str = LIB, extra=()) -> list:
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if not os.path.exists(nvcc):
        nvcc = "nvcc"
    return [nvcc, *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-fvisibility=hidden", "-shared", "-I" + os.path.join(ROOT, "include"),
            *extra, "-o", out, *SOURCES]


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile the library when it is missing or older than its sources."""
    if not force and os.path.exists(LIB):
        t = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) <= t for d in _deps()):
            return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = nvcc_command(tmp)
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build_library(force="--force" in sys.argv, verbose=True)
    print(LIB)
