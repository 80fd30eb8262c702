"""Builds libhashevict.so in-tree with nvcc for sm_103a (B300)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libhashevict.so")
SOURCES = [os.path.join(CSRC, "hashevict.cu"), os.path.join(CSRC, "he_noalloc.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")] + [
    os.path.join(INCLUDE, "hashevict.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared", "-Xptxas", "-warn-spills"]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library unless it is newer than every source."""
    if not force and os.path.exists(LIB):
        m = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) <= m for d in DEPS):
            return LIB
    cmd = ["nvcc", *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-o", LIB + ".tmp", *SOURCES]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
