"""Build libds4g.so in-tree for sm_103a (B300) with nvcc."""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(HERE, "libds4g.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(glob.glob(os.path.join(HERE, "csrc", "*.cu")))


def deps():
    root = os.path.dirname(HERE)
    return sources() + glob.glob(os.path.join(HERE, "csrc", "*.cuh")) + [os.path.join(root, "include", "ds4g.h")]


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(SO):
        t = os.path.getmtime(SO)
        if all(os.path.getmtime(d) <= t for d in deps()):
            return SO
    cmd = ["nvcc", "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
           "-o", SO, *sources()]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.check_call(cmd)
    return SO


if __name__ == "__main__":
    build(force=True, verbose="-v" in sys.argv)
    print(SO)
