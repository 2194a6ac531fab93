"""Build libfp8bs.so in-tree with nvcc for sm_103a (no JIT cache, no torch extension)."""
from __future__ import annotations

import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libfp8bs.so")
SRC = os.path.join(HERE, "csrc", "fp8bs.cu")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-shared", "-Xcompiler", "-fPIC",
    "-cudart", "shared",
    "-Xlinker", "-rpath=/usr/local/cuda/lib64",
]


def sources():
    return glob.glob(os.path.join(HERE, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*.h"))


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if force or stale():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [NVCC, *FLAGS, "-o", tmp, SRC]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.check_call(cmd)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
