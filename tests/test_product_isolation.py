"""The product path and the oracle stay apart: the package never imports the oracle (so
no call can fall back to the CPU), the kernels include nothing of it, the oracle uses
nothing of the package, and the binding fails loudly when the CUDA library is missing."""

import ast
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "quantized_moe_grouped_route_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _py_imports(path):
    tree = ast.parse(open(path).read())
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            names.add(node.module.split(".")[0])
    return names


def _files(d, exts):
    for dp, _, fs in os.walk(d):
        if "_build" in dp or "__pycache__" in dp:
            continue
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(dp, f)


def test_package_never_imports_the_oracle():
    for f in _files(PKG, (".py",)):
        assert "oracle" not in _py_imports(f), f


def test_kernels_include_nothing_of_the_oracle():
    for f in _files(PKG, (".cu", ".cuh", ".h", ".cpp")):
        for inc in re.findall(r'#include\s+[<"]([^>"]+)[>"]', open(f).read()):
            assert "oracle" not in inc and "qmoe_oracle" not in inc, (f, inc)


def test_oracle_uses_nothing_of_the_package():
    for f in _files(ORACLE, (".py",)):
        assert "quantized_moe_grouped_route_gb300" not in _py_imports(f), f
    for f in _files(ORACLE, (".c", ".h")):
        for inc in re.findall(r'#include\s+[<"]([^>"]+)[>"]', open(f).read()):
            assert inc.endswith(".h") and "/" not in inc and inc != "qmoe.h", (f, inc)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from quantized_moe_grouped_route_gb300 import qmoe
    monkeypatch.setattr(qmoe, "_lib", None)
    monkeypatch.setattr(qmoe, "LIB_PATH", str(tmp_path / "absent" / "libqmoe.so"))
    with pytest.raises(RuntimeError, match="missing"):
        qmoe.lib()
