"""The oracle is test infrastructure and the product never reaches it: a static
check (by syntax tree, no import of the modules checked) that

* no module of the package imports the oracle, and no CUDA or C source of the
  package includes a file of it;
* the oracle imports nothing of the package but the seeded input generators
  (which hold none of the method's arithmetic), and its C source includes no
  header of the library;
* in bench.py only the CPU legs touch it: `oracle_sample`, `cpu_baseline`, and
  the reference arm of `main`; no timing function of the GPU path names the
  oracle or those helpers;
* the binding raises when the library is missing instead of computing anything
  on the host."""
import ast
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "gated_delta_rule_166_b300")
ORACLE = os.path.join(ROOT, "oracle")
ORACLE_USERS = {"oracle_sample", "cpu_baseline"}


def _files(folder, exts):
    for dirpath, _, names in os.walk(folder):
        if "__pycache__" in dirpath or "_build" in dirpath:
            continue
        for n in sorted(names):
            if n.endswith(exts):
                yield os.path.join(dirpath, n)


def _imported_modules(tree):
    for n in ast.walk(tree):
        if isinstance(n, ast.Import):
            yield from (a.name for a in n.names)
        elif isinstance(n, ast.ImportFrom) and n.module:
            yield n.module
        elif isinstance(n, ast.Call) and getattr(n.func, "attr", getattr(n.func, "id", "")) in (
                "import_module", "__import__") and n.args and isinstance(n.args[0], ast.Constant):
            yield str(n.args[0].value)


def _parse(path):
    with open(path) as f:
        return ast.parse(f.read(), filename=path)


def test_package_never_imports_the_oracle():
    pys = list(_files(PKG, (".py",)))
    assert pys
    for path in pys:
        mods = set(_imported_modules(_parse(path)))
        assert not any(m.split(".")[0] == "oracle" for m in mods), (path, sorted(mods))
    for path in _files(PKG, (".cu", ".cuh", ".h", ".cpp", ".c")):
        with open(path) as f:
            includes = re.findall(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', f.read(), flags=re.M)
        assert not any("oracle" in i for i in includes), (path, includes)


def test_oracle_uses_only_the_input_generators_of_the_package():
    for path in _files(ORACLE, (".py",)):
        for m in _imported_modules(_parse(path)):
            if m.split(".")[0] == "gated_delta_rule_166_b300":
                assert m == "gated_delta_rule_166_b300.inputs", (path, m)
    for path in _files(ORACLE, (".c", ".h")):
        with open(path) as f:
            includes = re.findall(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', f.read(), flags=re.M)
        assert not any("gdr2" in i and "oracle" not in i for i in includes), (path, includes)


def _names(node):
    for n in ast.walk(node):
        if isinstance(n, ast.Name):
            yield n.id
        elif isinstance(n, ast.Attribute):
            yield n.attr


def test_bench_touches_the_oracle_only_in_its_cpu_legs():
    tree = _parse(os.path.join(ROOT, "bench.py"))
    # no module-level import of it
    top = [m for stmt in tree.body if isinstance(stmt, (ast.Import, ast.ImportFrom))
           for m in _imported_modules(stmt)]
    assert "oracle" not in top
    funcs = [f for f in ast.walk(tree) if isinstance(f, ast.FunctionDef)]
    assert {f.name for f in funcs} >= ORACLE_USERS | {"main"}
    for f in funcs:
        if f.name in ORACLE_USERS or f.name == "main":
            continue
        used = set(_names(f)) & ({"oracle"} | ORACLE_USERS)
        assert not used, (f.name, used)
    # in main: the oracle import sits under `if args.impl == "reference"`, and the
    # cpu baseline is called only where the flags ask for it
    main = next(f for f in funcs if f.name == "main")
    for n in ast.walk(main):
        if isinstance(n, ast.Import) and any(a.name == "oracle" for a in n.names):
            parents = [p for p in ast.walk(main) if isinstance(p, ast.If) and n in ast.walk(p)]
            assert any("reference" in ast.unparse(p.test) for p in parents), ast.unparse(n)


def test_binding_raises_without_the_library(monkeypatch, tmp_path):
    from gated_delta_rule_166_b300 import _lib

    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(_lib.GDR2LibraryError):
        _lib.lib()
    with pytest.raises(_lib.GDR2LibraryError):
        _lib.gdr2_version()
