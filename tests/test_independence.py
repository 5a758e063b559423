"""The oracle and the CUDA path share no code: the package never imports the
oracle, the oracle never imports the package, its native library or the
input generators, and bench.py imports the oracle only in its CPU-timing
functions (the CPU baseline and the reference arm)."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "gemm_epilogue_transformer_bf16_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "__pycache__" in d or "_build" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom) and node.module:
            yield node.module


def test_package_never_imports_the_oracle():
    for f in _files(PKG, (".py",)):
        assert not any(m.split(".")[0] == "oracle" for m in _imports(f)), f
    for f in _files(PKG, (".cu", ".cuh", ".h", ".cpp")):
        assert not re.search(r"#\s*include\s*[<\"][^>\"]*oracle", open(f).read()), f


def test_oracle_never_imports_the_product():
    banned = {"gemm_epilogue_transformer_bf16_gb300", "synth", "ctypes", "bench"}
    for f in _files(ORACLE, (".py",)):
        mods = {m.split(".")[0] for m in _imports(f)}
        assert not (mods & banned), (f, mods & banned)
        assert "libcoda" not in open(f).read(), f


def test_bench_imports_the_oracle_only_for_cpu_timing():
    path = os.path.join(ROOT, "bench.py")
    tree = ast.parse(open(path).read(), filename=path)
    users = set()

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            name = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            if isinstance(child, ast.ImportFrom) and child.module and child.module.split(".")[0] == "oracle":
                users.add(fn)
            if isinstance(child, ast.Import) and any(a.name.split(".")[0] == "oracle" for a in child.names):
                users.add(fn)
            visit(child, name)
    visit(tree, None)
    assert users == {"oracle_sample_timing", "oracle_workload_timings"}, users
