"""The product path never reaches the oracle and never falls back to the CPU:
the package imports nothing from oracle/, bench.py imports it only in its
CPU-oracle leg, and the binding refuses to import when the CUDA library has
not been built (no GPU needed)."""
import ast
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "nvfp4_mixture_experts_expert_gb300")


def _oracle_imports(tree):
    """(enclosing function name or None, line) of every import that names oracle."""
    found = []

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            f = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else func
            if isinstance(child, ast.Import) and any(a.name.split(".")[0] == "oracle" for a in child.names):
                found.append((func, child.lineno))
            elif isinstance(child, ast.ImportFrom) and (child.module or "").split(".")[0] == "oracle":
                found.append((func, child.lineno))
            visit(child, f)

    visit(tree, None)
    return found


def test_package_never_imports_the_oracle():
    for name in sorted(os.listdir(PKG)):
        if name.endswith(".py"):
            with open(os.path.join(PKG, name)) as f:
                tree = ast.parse(f.read())
            assert not _oracle_imports(tree), name


def test_bench_imports_the_oracle_only_in_its_cpu_oracle_leg():
    with open(os.path.join(ROOT, "bench.py")) as f:
        found = _oracle_imports(ast.parse(f.read()))
    assert found, "the CPU-oracle leg imports the oracle"
    assert {func for func, _ in found} <= {"oracle_prepare", "oracle_piece", "oracle_side_baselines"}


def test_binding_import_fails_loudly_without_the_library(tmp_path):
    dst = tmp_path / "nvfp4_mixture_experts_expert_gb300"
    shutil.copytree(PKG, dst, ignore=shutil.ignore_patterns("*.so", "_build", "__pycache__", "csrc"))
    assert not (dst / "libnvfp4moe.so").exists()
    r = subprocess.run([sys.executable, "-c", "import nvfp4_mixture_experts_expert_gb300.binding"],
                       cwd=tmp_path, env={**os.environ, "PYTHONPATH": str(tmp_path)}, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libnvfp4moe.so is missing" in r.stderr
