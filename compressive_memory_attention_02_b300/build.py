"""Build liblinattn.so (all CUDA sources of csrc/) for sm_103a with nvcc, and the
checked library liblinattn_checked.so (the same sources with LA_CHECKS=1: device-side
bounds checks that report through the status word; loaded when LA_CHECKED=1).

The libraries are built in-tree, next to this file, so that they ship with the
source tree; nothing is installed elsewhere.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "liblinattn.so")
LIB_CHECKED = os.path.join(HERE, "liblinattn_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-diag-suppress", "177"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def deps():
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))) + [
        os.path.join(os.path.dirname(HERE), "include", "linattn.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in deps())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB
    if not force and up_to_date(lib):
        return lib
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, *FLAGS, *(["-DLA_CHECKS=1"] if checked else []), "-o", tmp, *sources()]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), file=sys.stderr)
    subprocess.check_call(cmd)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
