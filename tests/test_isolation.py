"""The product path and the oracle stay apart, and the product has no CPU
fallback (CPU only; nothing here launches a kernel).

* No file of the package (Python binding, CUDA sources) imports or includes
  the oracle, and no oracle file uses the package or its CUDA sources.
* bench.py imports the oracle only inside its CPU-baseline functions (the
  reference arm calls those); __graft_entry__.py only in build() (compiling
  the checker) and smoke().
* Without its library the binding raises instead of computing, and its
  entry points refuse host tensors.
"""
import ast
import os
import re

import pytest
import torch

from fp8_fine_grained_22_b300 import fp8fg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fp8_fine_grained_22_b300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for dirpath, _, names in os.walk(top):
        if "__pycache__" in dirpath:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(dirpath, n)


def test_package_never_uses_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b|#\s*include\s*[<\"].*oracle)", re.M)
    hits = [p for p in _files(PKG, (".py", ".cu", ".cuh", ".h")) if pat.search(open(p).read())]
    assert not hits, hits


def test_oracle_never_uses_the_package():
    pat = re.compile(r"fp8_fine_grained_22_b300|\bcsrc\b|quant_math|fp8fg\.h|libfp8fg")
    hits = [p for p in _files(ORACLE, (".py", ".c", ".h")) if pat.search(open(p).read())]
    assert not hits, hits


def _functions_importing_oracle(path):
    tree = ast.parse(open(path).read())
    found = set()
    top_level = []
    for node in tree.body:
        for sub in ast.walk(node):
            is_import = (isinstance(sub, ast.Import) and any(a.name.split(".")[0] == "oracle"
                                                            for a in sub.names)) or \
                        (isinstance(sub, ast.ImportFrom) and (sub.module or "").split(".")[0] == "oracle")
            if is_import:
                if isinstance(node, ast.FunctionDef):
                    found.add(node.name)
                else:
                    top_level.append(sub.lineno)
    return found, top_level


def test_bench_and_entry_points_use_the_oracle_only_where_allowed():
    found, top = _functions_importing_oracle(os.path.join(ROOT, "bench.py"))
    assert not top, "bench.py imports the oracle at module level (lines %s)" % top
    assert found and all(f.startswith("cpu_baseline") for f in found), found
    found, top = _functions_importing_oracle(os.path.join(ROOT, "__graft_entry__.py"))
    assert not top and found <= {"build", "smoke"}, (found, top)


def test_binding_raises_without_its_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fp8fg, "_lib", None)
    monkeypatch.setattr(fp8fg, "LIB_PATH", str(tmp_path / "libfp8fg.so"))
    monkeypatch.setattr(fp8fg, "_build", lambda *a, **k: None)
    with pytest.raises(RuntimeError, match="missing"):
        fp8fg.lib()


def test_entry_points_refuse_host_tensors():
    x = torch.zeros((4, 128), dtype=torch.bfloat16)
    w = torch.zeros((128, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fp8fg.fp8_quant_act_1x128(x)
    with pytest.raises(ValueError):
        fp8fg.fp8_quant_weight_128x128(w)
    with pytest.raises(ValueError):
        fp8fg.fp8_quant_fprop_operands(x, w)
    q = torch.zeros((4, 128), dtype=torch.uint8)
    with pytest.raises(ValueError):
        fp8fg.fp8_gemm_blockscaled(q, torch.ones((1, 4)), q, torch.ones((1, 1)))
