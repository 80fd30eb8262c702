"""Builds libhashevict.so in-tree with nvcc for sm_103a (B300)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libhashevict.so")
# the same library with the device-side bounds checks of the debug build
DEBUG_LIB = os.path.join(PKG, "libhashevict_debug.so")
SOURCES = [os.path.join(CSRC, "hashevict.cu"), os.path.join(CSRC, "he_noalloc.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")] + [
    os.path.join(INCLUDE, "hashevict.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared", "-Xptxas", "-warn-spills"]


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile the library (with debug: the bounds-checked build) unless it is
    newer than every source."""
    out = DEBUG_LIB if debug else LIB
    if not force and os.path.exists(out):
        m = os.path.getmtime(out)
        if all(os.path.getmtime(d) <= m for d in DEPS):
            return out
    cmd = ["nvcc", *NVCC_FLAGS, *(["-DHE_DEBUG"] if debug else []), "-I", INCLUDE, "-I", CSRC,
           "-o", out + ".tmp", *SOURCES]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
    print(build(force=True, verbose=True, debug=True))
