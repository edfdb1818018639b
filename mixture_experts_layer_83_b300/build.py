"""Build the in-tree shared library ``libmoe_b300.so`` (sm_103a only) with nvcc."""
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libmoe_b300.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
         "-Xptxas", "-warn-spills", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def deps():
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) +
                              glob.glob(os.path.join(CSRC, "*.h")) +
                              [os.path.join(ROOT, "include", "moe_layer.h")])


def up_to_date(lib, inputs):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in inputs)


def build(force=False, verbose=False, extra=()):
    if not force and up_to_date(LIB, deps()):
        return LIB
    cmd = [NVCC] + ARCH + FLAGS + list(extra) + ["-o", LIB] + sources()
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True, extra=sys.argv[1:])
