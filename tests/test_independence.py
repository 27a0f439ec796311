"""The oracle and the CUDA path share nothing: no module of the package
imports the oracle, no CUDA source includes an oracle file, and the oracle
includes no header, table or module of the package. bench.py may use the
oracle only in its CPU legs (the timed CPU baseline and the reference arm)."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "quantised_linear_layers_gb300")
CSRC = os.path.join(PKG, "csrc")
ORACLE = os.path.join(ROOT, "oracle")


def _imports(path):
    tree = ast.parse(open(path).read())
    out = []
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            out += [(a.name, node) for a in node.names]
        elif isinstance(node, ast.ImportFrom):
            out.append((node.module or "", node))
    return tree, out


def test_package_never_imports_the_oracle():
    for f in os.listdir(PKG):
        if f.endswith(".py"):
            _, imps = _imports(os.path.join(PKG, f))
            assert not [m for m, _ in imps if m.split(".")[0] == "oracle"], f


def test_cuda_sources_include_nothing_of_the_oracle():
    for f in os.listdir(CSRC):
        if f.endswith((".cu", ".cuh", ".h")):
            src = open(os.path.join(CSRC, f)).read()
            for inc in re.findall(r'#include\s+"([^"]+)"', src):
                assert "oracle" not in inc, (f, inc)


def test_oracle_includes_nothing_of_the_package():
    for f in os.listdir(ORACLE):
        p = os.path.join(ORACLE, f)
        if f.endswith(".c"):
            incs = re.findall(r'#include\s+[<"]([^>"]+)[>"]', open(p).read())
            assert all(i in ("math.h", "stdint.h", "string.h", "stdlib.h", "omp.h") for i in incs), incs
        elif f.endswith(".py"):
            _, imps = _imports(p)
            mods = {m.split(".")[0] for m, _ in imps}
            assert "quantised_linear_layers_gb300" not in mods, f
            assert not (mods & {"torch", "triton"}), (f, mods)


def test_bench_uses_the_oracle_only_in_its_cpu_legs():
    tree, imps = _imports(os.path.join(ROOT, "bench.py"))
    owners = {}
    for node in ast.walk(tree):
        if isinstance(node, (ast.FunctionDef, ast.ClassDef)):
            for sub in ast.walk(node):
                if isinstance(sub, (ast.Import, ast.ImportFrom)):
                    owners.setdefault(id(sub), node.name)
    for mod, node in imps:
        if mod.split(".")[0] == "oracle":
            # the CPU legs: the sample of the headline workload and the
            # oracle timings of the smaller configurations
            assert owners.get(id(node)) in ("CpuOracleSample", "cpu_baselines"), owners.get(id(node))


def test_entry_uses_the_oracle_only_to_build_and_check():
    tree, imps = _imports(os.path.join(ROOT, "__graft_entry__.py"))
    owners = {}
    for node in ast.walk(tree):
        if isinstance(node, ast.FunctionDef):
            for sub in ast.walk(node):
                if isinstance(sub, (ast.Import, ast.ImportFrom)):
                    owners.setdefault(id(sub), node.name)
    for mod, node in imps:
        if mod.split(".")[0] == "oracle":
            assert owners.get(id(node)) in ("build", "smoke"), owners.get(id(node))
