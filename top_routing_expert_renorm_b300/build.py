"""Build libmoe.so (the C-ABI MoE layer library) in-tree for sm_103a with nvcc."""

import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libmoe.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in sources())


def nvcc_cmd(out, extra=()):
    return [NVCC, "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
            "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64", "-I", INCLUDE,
            *extra, "-o", out, os.path.join(CSRC, "moe_api.cu")]


def build(force=False, verbose=False):
    """Compile the library when missing or older than any source; return its path."""
    if not force and not stale():
        return LIB
    tmp = LIB + ".tmp"
    extra = ["-Xptxas", "-v"] if verbose else []
    subprocess.run(nvcc_cmd(tmp, extra), check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
