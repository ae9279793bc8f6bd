"""The product path and the oracle are separate programs (no GPU needed).

* No module of the package imports the oracle, and no CUDA source includes
  anything from it.
* The built library neither defines nor needs an oracle symbol, and does not
  link the oracle's shared object.
* The oracle's C source includes nothing from the library.
* Without the built library the binding raises instead of computing anything
  another way.
"""
import ast
import os
import re
import subprocess

import pytest

from conftest import ROOT

PKG = os.path.join(ROOT, "quantized_moe_routed_gb300")
CSRC = os.path.join(PKG, "csrc")


def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom):
            yield node.module or ""


def test_package_never_imports_the_oracle():
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith(".py"):
                for mod in _imports(os.path.join(dirpath, f)):
                    assert mod.split(".")[0] != "oracle", f"{f} imports {mod}"


def test_sources_do_not_cross():
    for f in os.listdir(CSRC):
        src = open(os.path.join(CSRC, f)).read()
        assert not re.search(r'#include\s*[<"][^>"]*oracle', src), f
    src = open(os.path.join(ROOT, "oracle", "moe_oracle.c")).read()
    for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', src):
        assert inc in ("math.h", "stdint.h", "stdlib.h", "string.h", "omp.h"), inc


def test_library_has_no_oracle_symbols():
    from quantized_moe_routed_gb300 import build as libbuild
    lib = libbuild.build()
    out = subprocess.run(["nm", "-D", lib], check=True, capture_output=True, text=True).stdout
    assert "oracle" not in out
    needed = subprocess.run(["readelf", "-d", lib], check=True, capture_output=True, text=True).stdout
    assert "moe_oracle" not in needed


def test_missing_library_raises(monkeypatch):
    from quantized_moe_routed_gb300 import MoeError, binding
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(MoeError) as ei:
        binding.load_library(os.path.join(ROOT, "no_such_dir", "libmoe_nvfp4.so"))
    assert "no fallback" in str(ei.value)
