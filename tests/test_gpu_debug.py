"""The bounds-checked build (libfp8bs_debug.so, FP8BS_DEBUG) on small odd shapes of
every kernel family: no access site's index leaves its extent, and the results still
match the oracle.  Runs tests/debug_shapes.py in a child process, because a process
loads one build of the library."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_debug_build_on_odd_shapes():
    env = dict(os.environ, FP8BS_LIBRARY="debug")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_shapes.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "debug ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


def test_debug_library_exports_the_abi():
    """CPU: the bounds-checked twin exports every symbol of the header and says it is the debug build."""
    import ctypes
    from fp8_fine_grained_27_b300 import binding, build
    lib = ctypes.CDLL(build.LIB_DEBUG)
    for name in binding.EXPORTS:
        assert hasattr(lib, name), name
    assert lib.fp8bs_debug_build() == 1
    assert ctypes.CDLL(build.LIB).fp8bs_debug_build() == 0
