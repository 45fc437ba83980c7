"""The oracle and the CUDA path stay independent, checked statically.

- The product package (binding, build script, CUDA/C++ sources and the
  public header) names nothing of the oracle.
- The oracle imports nothing of the product package and no local module.
- The shared input generator imports neither.
- bench.py imports the oracle only inside functions (its CPU-baseline and
  reference legs), never at module level, so the timed GPU path cannot reach
  it.
"""

import ast
import glob
import os

from conftest import ROOT

PKG = os.path.join(ROOT, "mxfp8_block_scaled_inv_gb300")


def _imports(path):
    """(module names imported at module level, module names imported anywhere)."""
    tree = ast.parse(open(path).read(), filename=path)
    top, anywhere = set(), set()

    def names(node):
        if isinstance(node, ast.Import):
            return {a.name.split(".")[0] for a in node.names}
        if isinstance(node, ast.ImportFrom):
            return {(node.module or "").split(".")[0]} if node.level == 0 else {"."}
        return set()

    for node in tree.body:
        top |= names(node)
    for node in ast.walk(tree):
        anywhere |= names(node)
    return top, anywhere


def test_product_sources_name_nothing_of_the_oracle():
    files = glob.glob(os.path.join(PKG, "*.py")) + glob.glob(os.path.join(PKG, "csrc", "*"))
    files += glob.glob(os.path.join(ROOT, "include", "*.h"))
    files = [f for f in files if os.path.isfile(f) and not f.endswith((".so", ".o"))]
    assert files
    for f in files:
        text = open(f, errors="replace").read()
        assert "mx_oracle" not in text and "oracle/" not in text, f
        if f.endswith(".py"):
            assert "oracle" not in _imports(f)[1], f


def test_oracle_imports_no_local_module():
    for f in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        _, mods = _imports(f)
        assert not mods & {"mxfp8_block_scaled_inv_gb300", "workloads", "bench", "tests", "."}, f


def test_input_generator_imports_neither_side():
    _, mods = _imports(os.path.join(ROOT, "workloads", "__init__.py"))
    assert not mods & {"oracle", "mxfp8_block_scaled_inv_gb300"}


def test_bench_imports_the_oracle_only_inside_its_cpu_legs():
    path = os.path.join(ROOT, "bench.py")
    top, anywhere = _imports(path)
    assert "oracle" not in top
    assert "oracle" in anywhere  # the CPU-baseline / reference legs
    tree = ast.parse(open(path).read())
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            inner = {n.module for n in ast.walk(fn) if isinstance(n, ast.ImportFrom) and n.module}
            if "oracle" in inner:
                assert fn.name.startswith(("oracle_", "_oracle")), fn.name
