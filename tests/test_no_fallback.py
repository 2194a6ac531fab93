"""The product path has no CPU fallback: without libfp8bs.so the binding raises at first
use, and nothing in the package imports the oracle."""
import ast
import os

import pytest


def test_missing_library_raises(monkeypatch, tmp_path):
    from fp8_fine_grained_27_b300 import binding
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(ImportError):
        binding.lib()


def test_package_never_imports_the_oracle():
    root = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "fp8_fine_grained_27_b300")
    for name in os.listdir(root):
        if name.endswith(".py"):
            tree = ast.parse(open(os.path.join(root, name)).read())
            for node in ast.walk(tree):
                mods = []
                if isinstance(node, ast.Import):
                    mods = [a.name for a in node.names]
                elif isinstance(node, ast.ImportFrom) and node.module:
                    mods = [node.module]
                assert not any(m.split(".")[0] == "oracle" for m in mods), (name, mods)
