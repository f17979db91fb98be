"""Structural checks: the CPU oracle and the CUDA path share no code and do
not import each other, and the product path has no fallback when its
library is missing."""

import ast
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fp8_weight_only_nvfp4_gb300")
CSRC = os.path.join(PKG, "csrc")
ORACLE = os.path.join(ROOT, "oracle")


def _files(d, exts):
    out = []
    for base, dirs, files in os.walk(d):
        dirs[:] = [x for x in dirs if x not in ("__pycache__", "_build")]
        out += [os.path.join(base, f) for f in files if f.endswith(exts)]
    return out


def _py_imports(path):
    tree = ast.parse(open(path).read())
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.module:
            names.add(node.module.split(".")[0])
    return names


def test_oracle_includes_nothing_from_the_cuda_path():
    for f in _files(ORACLE, (".cpp", ".c", ".h", ".hpp")):
        src = open(f).read()
        for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', src):
            assert "csrc" not in inc and not inc.startswith("wqmm_") and "include/" not in inc, (f, inc)
    for f in _files(ORACLE, (".py",)):
        assert "fp8_weight_only_nvfp4_gb300" not in _py_imports(f), f


def test_cuda_path_includes_nothing_from_the_oracle():
    for f in _files(CSRC, (".cu", ".cuh", ".h")):
        src = open(f).read()
        for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', src):
            assert "oracle" not in inc, (f, inc)
    for f in _files(PKG, (".py",)):
        assert "oracle" not in _py_imports(f), f


def test_shared_input_module_holds_no_method_arithmetic():
    """workloads/ (the seeded generators both sides use) imports neither side."""
    for f in _files(os.path.join(ROOT, "workloads"), (".py",)):
        imps = _py_imports(f)
        assert "oracle" not in imps and "fp8_weight_only_nvfp4_gb300" not in imps, f


def test_product_path_raises_without_its_library(tmp_path, monkeypatch):
    import fp8_weight_only_nvfp4_gb300 as wq
    monkeypatch.setattr(wq, "_LIB_PATH", str(tmp_path / "libwqmm.so"))
    monkeypatch.setattr(wq, "_lib", None)
    with pytest.raises(ImportError):
        wq.lib()
