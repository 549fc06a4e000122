"""The CUDA path and the oracle share nothing, and only test code reaches the oracle.

Static checks over the sources (no build, no GPU):
* no module of the product package, and neither engine script, imports
  ``oracle``; ``bench.py`` does so only in its CPU-baseline and reference-arm
  functions, ``__graft_entry__`` only in ``build`` (compiling it) and
  ``smoke`` (checking against it);
* the oracle imports nothing from the product package, and its C source
  includes only its own header and the C library;
* the CUDA sources include nothing from ``oracle/``;
* the shared seeded-input module imports neither side.
"""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "w8a8_int8_quantized_i8_gb300"

ALLOWED_ORACLE_USERS = {
    "bench.py": {"_oracle_sample", "run_reference"},
    "__graft_entry__.py": {"build", "smoke"},
}


def _imports(tree):
    """(top-level module name, enclosing function names) for every import."""
    out = []

    def visit(node, funcs):
        for child in ast.iter_child_nodes(node):
            f = funcs
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)):
                f = funcs + (child.name,)
            if isinstance(child, ast.Import):
                out.extend((a.name.split(".")[0], f) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                if child.level:                       # relative: inside its own package
                    out.append(("." + (child.module or ""), f))
                else:
                    out.append(((child.module or "").split(".")[0], f))
            visit(child, f)

    visit(tree, ())
    return out


def _parse(path):
    with open(path) as fh:
        return ast.parse(fh.read(), path)


def test_product_package_never_imports_the_oracle():
    files = glob.glob(os.path.join(ROOT, PKG, "**", "*.py"), recursive=True)
    files.append(os.path.join(ROOT, "bench_engines.py"))
    assert len(files) > 5
    for path in files:
        for mod, _ in _imports(_parse(path)):
            assert mod != "oracle", path


def test_bench_and_entry_import_the_oracle_only_where_allowed():
    for name, allowed in ALLOWED_ORACLE_USERS.items():
        seen = set()
        for mod, funcs in _imports(_parse(os.path.join(ROOT, name))):
            if mod == "oracle":
                assert funcs and funcs[-1] in allowed, (name, funcs)
                seen.add(funcs[-1])
        assert seen == allowed, (name, seen)


def test_oracle_imports_nothing_from_the_product():
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        for mod, _ in _imports(_parse(path)):
            assert mod != PKG and not mod.startswith("."), (path, mod)
    allowed = {'"i8_oracle.h"', "<math.h>", "<stddef.h>", "<string.h>", "<omp.h>", "<stdint.h>"}
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.[ch]")):
        with open(path) as fh:
            incs = set(re.findall(r"^\s*#\s*include\s+(\S+)", fh.read(), re.M))
        assert incs <= allowed, (path, incs - allowed)


def test_cuda_sources_include_nothing_from_the_oracle():
    for path in glob.glob(os.path.join(ROOT, PKG, "csrc", "*")):
        with open(path) as fh:
            text = fh.read()
        for inc in re.findall(r"^\s*#\s*include\s+(\S+)", text, re.M):
            assert "oracle" not in inc, (path, inc)


def test_shared_input_module_imports_neither_side():
    mods = {m for m, _ in _imports(_parse(os.path.join(ROOT, PKG, "inputs.py")))}
    assert mods <= {"__future__", "dataclasses", "numpy", "torch"}, mods
