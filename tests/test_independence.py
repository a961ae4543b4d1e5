"""The oracle and the CUDA path share no code, and only the test harness
touches the oracle.  Checked statically on the sources (CPU only):

* no module of the package imports ``oracle``, and the oracle imports nothing
  of the package;
* the library is built from the package's own CUDA sources only;
* ``bench.py`` imports the oracle only inside its CPU-baseline and
  reference-arm functions, ``__graft_entry__`` only inside ``smoke()``;
* the binding refuses to run without the compiled library (no fallback).
"""
import ast
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "quantized_attention_gb300")

# bench.py functions that time the oracle (cpu_baseline leg, reference arm)
BENCH_ORACLE_FUNCS = {"_oracle_sample_worker", "sample_problem", "time_cpu_mode_baseline"}


def _imports(tree):
    """(module name, enclosing function name or None) for every import."""
    out = []

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            f = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else func
            if isinstance(child, ast.Import):
                out.extend((a.name, f) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                out.append(("." * child.level + (child.module or ""), f))
            visit(child, f)

    visit(tree, None)
    return out


def _parse(path):
    with open(path) as fh:
        return ast.parse(fh.read(), path)


def _py_files(d):
    for dirpath, _, files in os.walk(d):
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(dirpath, f)


def test_package_never_imports_the_oracle():
    for path in _py_files(PKG):
        for mod, _ in _imports(_parse(path)):
            assert not mod.split(".")[0] == "oracle", f"{path} imports {mod}"


def test_oracle_imports_nothing_of_the_package():
    for path in _py_files(os.path.join(ROOT, "oracle")):
        for mod, _ in _imports(_parse(path)):
            top = mod.lstrip(".").split(".")[0]
            assert top in ("", "__future__", "math", "numpy", "qattn_oracle"), f"{path} imports {mod}"


def test_library_sources_are_the_package_cuda_files():
    from quantized_attention_gb300 import build
    csrc = os.path.join(PKG, "csrc")
    for src in build.SOURCES:
        assert os.path.exists(os.path.join(csrc, src)), src
        with open(os.path.join(csrc, src)) as fh:
            for line in fh:
                if line.lstrip().startswith("#include"):
                    assert "oracle" not in line, f"{src}: {line.strip()}"


@pytest.mark.parametrize("name,allowed", [("bench.py", BENCH_ORACLE_FUNCS),
                                          ("__graft_entry__.py", {"smoke"})])
def test_oracle_imported_only_by_the_harness_functions(name, allowed):
    users = {f for mod, f in _imports(_parse(os.path.join(ROOT, name)))
             if mod.split(".")[0] == "oracle"}
    assert users and users <= allowed, f"{name}: oracle imported in {sorted(map(str, users))}"


def test_binding_fails_loudly_without_the_library(monkeypatch):
    from quantized_attention_gb300 import binding as qb
    monkeypatch.setattr(qb, "_lib", None)
    monkeypatch.setattr(qb, "_LIB_PATH", os.path.join(ROOT, "no-such-dir", "libqattn.so"))
    with pytest.raises(RuntimeError, match="missing"):
        qb.lib()
