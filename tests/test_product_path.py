"""The product path has no fallback (CPU only).

The library's kernels are the only compute path: importing the package with
its CUDA library missing must fail loudly rather than fall back to anything,
and no module of the package imports the fp64 oracle, which is test
infrastructure (only tests/, smoke() and bench.py's CPU-baseline and
reference arms may use it).
"""
from __future__ import annotations

import ast
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "full_gqa_attention_gb300")


def test_missing_library_fails_loudly(tmp_path):
    """A copy of the package without its built library cannot be imported."""
    shutil.copytree(PKG, tmp_path / "full_gqa_attention_gb300",
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    code = (
        "try:\n"
        "    import full_gqa_attention_gb300\n"
        "except ImportError as e:\n"
        "    print('ImportError:', e)\n"
        "else:\n"
        "    print('imported')\n"
    )
    env = dict(os.environ, PYTHONPATH=str(tmp_path))
    run = subprocess.run([sys.executable, "-c", code], cwd=str(tmp_path), env=env,
                         capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stderr
    assert run.stdout.startswith("ImportError:"), run.stdout
    assert "not built" in run.stdout


def _imported_modules(path: str) -> set[str]:
    tree = ast.parse(open(path).read(), filename=path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module:
            names.add(node.module.split(".")[0])
    return names


def test_package_never_imports_the_oracle():
    for name in sorted(os.listdir(PKG)):
        if name.endswith(".py"):
            assert "oracle" not in _imported_modules(os.path.join(PKG, name)), name


def test_bench_uses_the_oracle_only_in_its_baseline_arms():
    """bench.py imports the oracle only inside the functions that time it."""
    path = os.path.join(ROOT, "bench.py")
    tree = ast.parse(open(path).read(), filename=path)
    for node in tree.body:   # no module-level import
        if isinstance(node, (ast.Import, ast.ImportFrom)):
            mods = ([a.name for a in node.names] if isinstance(node, ast.Import)
                    else [node.module or ""])
            assert not any(m.split(".")[0] == "oracle" for m in mods)
    users = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.FunctionDef):
            for sub in ast.walk(node):
                if isinstance(sub, ast.Import) and any(a.name == "oracle" for a in sub.names):
                    users.add(node.name)
    assert users and all(u.startswith("oracle_") for u in users), users


def test_cuda_sources_do_not_include_the_oracle():
    csrc = os.path.join(PKG, "csrc")
    for name in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, name)).read()
        assert "spark_oracle" not in text and "oracle/" not in text, name


def test_oracle_shares_no_code_with_the_cuda_path():
    """The oracle includes only the C standard library and imports neither the
    package nor anything of the CUDA path; the two meet only in the tests."""
    odir = os.path.join(ROOT, "oracle")
    std = {"math.h", "stdint.h", "stdlib.h", "string.h", "stdio.h", "float.h", "omp.h"}
    for name in sorted(os.listdir(odir)):
        path = os.path.join(odir, name)
        if name.endswith(".c"):
            for line in open(path):
                if line.lstrip().startswith("#include"):
                    header = line.split("#include", 1)[1].strip().strip("<>\"")
                    assert header in std, (name, header)
        elif name.endswith(".py"):
            mods = _imported_modules(path)
            assert "full_gqa_attention_gb300" not in mods and "workloads" not in mods, (name, mods)
