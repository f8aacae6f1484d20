"""The oracle and the CUDA path share no code, and the product path never
reaches the oracle: checked on the sources, without a GPU.

* nothing in the package (Python or CUDA) or in include/ imports, includes or
  names the oracle's module, header or library;
* the oracle imports nothing of the package and includes nothing of csrc/;
* in bench.py the oracle is imported only inside the functions that time it
  (the CPU baseline and the reference arm); __graft_entry__ only in build()
  (which compiles it) and smoke() (which checks against it).
"""
import ast
import glob
import os
import re

from conftest import ROOT

PKG = os.path.join(ROOT, "mhc_residual_boundary_gb300")


def _files(*patterns):
    out = []
    for p in patterns:
        out += glob.glob(os.path.join(ROOT, p), recursive=True)
    return sorted(f for f in out if "__pycache__" not in f)


def _python_imports(path):
    tree = ast.parse(open(path).read())
    found = []
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            found += [(a.name, node) for a in node.names]
        elif isinstance(node, ast.ImportFrom):
            found.append((node.module or "", node))
    return tree, found


def test_product_sources_never_reach_the_oracle():
    for f in _files("mhc_residual_boundary_gb300/**/*.py"):
        _, imports = _python_imports(f)
        assert not any(name.split(".")[0] == "oracle" for name, _ in imports), f
    for f in _files("mhc_residual_boundary_gb300/**/*.cu", "mhc_residual_boundary_gb300/**/*.cuh",
                    "include/*.h"):
        text = open(f).read()
        assert not re.search(r'#include\s*[<"][^>"]*oracle', text), f
        assert "mhc_oracle" not in text and "liboracle" not in text, f


def test_oracle_takes_nothing_from_the_package():
    for f in _files("oracle/*.py"):
        _, imports = _python_imports(f)
        assert not any(name.startswith("mhc_residual_boundary_gb300") for name, _ in imports), f
    for f in _files("oracle/*.c", "oracle/*.h"):
        includes = re.findall(r'#include\s*[<"]([^>"]+)[>"]', open(f).read())
        assert all(i in ("mhc_oracle.h", "math.h", "stdlib.h", "string.h", "stddef.h", "stdint.h")
                   for i in includes), (f, includes)


def _functions_importing_oracle(path):
    tree, _ = _python_imports(path)
    where = set()

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)):
                visit(child, child.name)
            else:
                if isinstance(child, ast.Import) and any(a.name.split(".")[0] == "oracle" for a in child.names):
                    where.add(func)
                if isinstance(child, ast.ImportFrom) and (child.module or "").split(".")[0] == "oracle":
                    where.add(func)
                visit(child, func)

    visit(tree, None)
    return where


def test_bench_and_entry_import_the_oracle_only_where_allowed():
    bench = _functions_importing_oracle(os.path.join(ROOT, "bench.py"))
    assert bench and bench <= {"oracle_tokens_per_s", "run_reference", "cpu_baseline"}, bench
    entry = _functions_importing_oracle(os.path.join(ROOT, "__graft_entry__.py"))
    assert entry <= {"build", "smoke"}, entry
