"""The oracle stays test infrastructure: the product package and the CUDA sources never
refer to it, and bench.py reaches it only from its CPU-baseline / reference-arm sampler.
Static checks on the sources (CPU only)."""
from __future__ import annotations

import ast
import glob
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_MODULES = ("oracle", "tests.gpu_util", "tests.oracle_pins", "tests.projection_pins")


def _imports(path):
    """(module, enclosing function or None) for every import statement of a Python file."""
    tree = ast.parse(open(path).read(), path)
    out = []

    def visit(node, fn):
        for ch in ast.iter_child_nodes(node):
            f = ch.name if isinstance(ch, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            if isinstance(ch, ast.Import):
                out.extend((a.name, f) for a in ch.names)
            elif isinstance(ch, ast.ImportFrom):
                mod = ch.module or ""
                out.append((mod, f))
                out.extend((f"{mod}.{a.name}" if mod else a.name, f) for a in ch.names)
            visit(ch, f)
    visit(tree, None)
    return out


def _is_oracle(mod):
    return any(mod == m or mod.startswith(m + ".") for m in ORACLE_MODULES)


def test_package_never_imports_the_oracle():
    for path in glob.glob(os.path.join(ROOT, "causal_attention_gb300", "**", "*.py"), recursive=True):
        bad = [m for m, _ in _imports(path) if _is_oracle(m)]
        assert not bad, f"{path} imports {bad}"


def test_cuda_sources_never_refer_to_the_oracle():
    for path in glob.glob(os.path.join(ROOT, "causal_attention_gb300", "csrc", "*")) + \
            glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(path).read()
        assert "oracle" not in src.lower(), path


def test_bench_reaches_the_oracle_only_from_the_cpu_sampler():
    uses = [(m, f) for m, f in _imports(os.path.join(ROOT, "bench.py")) if _is_oracle(m)]
    assert uses, "the CPU baseline samples the oracle"
    assert all(f == "oracle_sample" for _, f in uses), uses


def test_importing_bench_loads_no_oracle_module():
    code = ("import sys; sys.path.insert(0, %r); import bench; "
            "bad = [m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')]; "
            "assert not bad, bad" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
