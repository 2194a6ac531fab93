"""Build the in-tree libraries with nvcc for sm_103a (no JIT cache, no torch extension):
libfp8bs.so (the release build) and libfp8bs_debug.so (the same source compiled
with FP8BS_DEBUG: every kernel access site checks its index and records a failure
instead of touching memory; see fp8bs_debug_site in include/fp8bs.h)."""
from __future__ import annotations

import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libfp8bs.so")
LIB_DEBUG = os.path.join(HERE, "libfp8bs_debug.so")
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


def stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in sources())


def _compile(lib: str, extra: list[str], force: bool, verbose: bool) -> str:
    if force or stale(lib):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [NVCC, *FLAGS, *extra, "-o", tmp, SRC]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.check_call(cmd)
        os.replace(tmp, lib)
    return lib


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Build the release library (and, with debug=True, the bounds-checked one too);
    returns the release library's path."""
    if debug:
        _compile(LIB_DEBUG, ["-DFP8BS_DEBUG"], force, verbose)
    return _compile(LIB, [], force, verbose)


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
