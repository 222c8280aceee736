"""The oracle is test infrastructure: the product package (Python binding,
CUDA sources, headers) neither imports nor includes anything from oracle/,
and bench.py reaches it only through its CPU-baseline helper (the reference
arm and the cpu_baseline leg). The oracle in turn uses nothing of the
package's arithmetic."""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "sparse_moe_transformer_limited_b300")


def _files(top, exts):
    for d, _, names in os.walk(top):
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def _imported_modules(path):
    tree = ast.parse(open(path).read())
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name, node
        elif isinstance(node, ast.ImportFrom) and node.module:
            yield node.module, node


def test_package_python_does_not_import_the_oracle():
    for f in _files(PKG, (".py",)):
        for mod, _ in _imported_modules(f):
            assert not mod.split(".")[0] in ("oracle", "beam_oracle"), (f, mod)


def test_package_native_sources_do_not_reference_the_oracle():
    for f in list(_files(PKG, (".cu", ".cuh", ".h", ".cpp"))) + list(
            _files(os.path.join(ROOT, "include"), (".h",))):
        text = open(f, encoding="utf-8").read()
        assert "oracle" not in text.lower(), f


def test_bench_reaches_the_oracle_only_through_its_cpu_baseline_helper():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    users = []
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, (ast.Import, ast.ImportFrom)):
                    names = ([a.name for a in node.names] if isinstance(node, ast.Import)
                             else [node.module or ""])
                    if any(n.split(".")[0] == "oracle" for n in names):
                        users.append(fn.name)
    # no module-level import either
    for node in tree.body:
        if isinstance(node, (ast.Import, ast.ImportFrom)):
            names = ([a.name for a in node.names] if isinstance(node, ast.Import)
                     else [node.module or ""])
            assert not any(n.split(".")[0] == "oracle" for n in names)
    assert users == ["oracle_sample"], users


def test_oracle_does_not_use_the_package():
    for f in _files(os.path.join(ROOT, "oracle"), (".py",)):
        for mod, _ in _imported_modules(f):
            assert not mod.startswith("sparse_moe_transformer_limited_b300"), (f, mod)
