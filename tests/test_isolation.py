"""The oracle and the CUDA path share nothing, and the product never runs the
oracle.  Read from the sources: no file of the package (Python, CUDA, the
header) imports, includes, loads or names the oracle's code; the oracle
imports nothing from the package and includes no header of it; the only
places outside the tests that import the oracle are the smoke check and
bench.py's host-side (CPU baseline, reference arm) functions."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "moe_decode_tail_gb300")


def _files(top, exts):
    for d, dirs, fs in os.walk(top):
        dirs[:] = [x for x in dirs if x not in ("__pycache__", "_build", "build")]
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(d, f)


def _imports(path):
    tree = ast.parse(open(path).read())
    out = []
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            out += [a.name.split(".")[0] for a in node.names]
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            out.append(node.module.split(".")[0])
    return out


def test_package_never_imports_or_links_the_oracle():
    for f in _files(PKG, (".py",)):
        assert "oracle" not in _imports(f), f
    for f in list(_files(PKG, (".cu", ".cuh", ".h", ".cpp"))) + list(_files(os.path.join(ROOT, "include"), (".h",))):
        text = open(f).read()
        assert not re.search(r"#\s*include\s*[<\"][^>\"]*oracle", text), f
        assert "oracle_" not in text, f  # no oracle symbol is declared or called


def test_oracle_takes_nothing_from_the_package():
    for f in _files(os.path.join(ROOT, "oracle"), (".py",)):
        assert "moe_decode_tail_gb300" not in _imports(f), f
    src = open(os.path.join(ROOT, "oracle", "moe_tail_oracle.c")).read()
    includes = re.findall(r"#\s*include\s*[<\"]([^>\"]+)[>\"]", src)
    assert set(includes) <= {"math.h", "stdint.h", "stdlib.h", "string.h"}, includes


def test_oracle_imported_only_in_the_allowed_places():
    # __graft_entry__: build() compiles it, smoke() checks against it; bench.py:
    # only inside its host-side timing functions, never at module level
    assert "oracle" in _imports(os.path.join(ROOT, "__graft_entry__.py"))
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    top = [n for n in tree.body if isinstance(n, (ast.Import, ast.ImportFrom))]
    assert all("oracle" not in [a.name for a in n.names] and getattr(n, "module", None) != "oracle" for n in top)
    users = set()
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, ast.Import) and any(a.name == "oracle" for a in node.names):
                    users.add(fn.name)
    assert users == {"oracle_token_times", "oracle_parallel_times"}, users


def test_bench_runs_the_oracle_only_for_the_cpu_baseline_and_the_reference_arm():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    callers = set()
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if (isinstance(node, ast.Call) and isinstance(node.func, ast.Name)
                        and node.func.id in ("oracle_token_times", "oracle_parallel_times")):
                    callers.add(fn.name)
    assert callers == {"cpu_baseline", "reference_arm"}, callers
