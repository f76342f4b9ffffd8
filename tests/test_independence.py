"""The oracle and the CUDA path share no code and neither imports the other.

Checked statically: no module of the package imports ``oracle``; no oracle
module imports the package (inputs reach the oracle as arrays from the
tests); the C sources of each side include nothing from the other; and the
only other importers of the oracle are the places allowed to run it:
``bench.py``'s oracle timing, ``__graft_entry__.smoke()``, and
``__graft_entry__.build()`` (which compiles it)."""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "zero_partitioned_mixed_replica_gb300"


def _imports(path):
    """(top-level module name, enclosing function or None) of every import."""
    tree = ast.parse(open(path).read(), path)
    out = []

    def visit(node, func):
        for ch in ast.iter_child_nodes(node):
            f = ch.name if isinstance(ch, (ast.FunctionDef, ast.AsyncFunctionDef)) else func
            if isinstance(ch, ast.Import):
                out.extend((a.name.split(".")[0], func) for a in ch.names)
            elif isinstance(ch, ast.ImportFrom) and ch.module and ch.level == 0:
                out.append((ch.module.split(".")[0], func))
            visit(ch, f)

    visit(tree, None)
    return out


def test_package_never_imports_the_oracle():
    files = glob.glob(os.path.join(ROOT, PKG, "**", "*.py"), recursive=True)
    assert files
    for p in files:
        assert "oracle" not in [m for m, _ in _imports(p)], p


def test_oracle_never_imports_the_package():
    files = glob.glob(os.path.join(ROOT, "oracle", "*.py"))
    assert files
    for p in files:
        mods = [m for m, _ in _imports(p)]
        assert PKG not in mods and "tests" not in mods, p


def test_oracle_is_run_only_where_allowed():
    allowed = {"bench.py": {"oracle_timing"}, "__graft_entry__.py": {"build", "smoke"}}
    for name, funcs in allowed.items():
        seen = set()
        for mod, func in _imports(os.path.join(ROOT, name)):
            if mod == "oracle":
                assert func in funcs, (name, func)
                seen.add(func)
        assert seen == funcs, (name, seen)      # the scan did find them


def test_c_sources_include_nothing_from_the_other_side():
    inc = re.compile(r'^\s*#\s*include\s*([<"])([^>"]+)[>"]', re.M)
    for p in glob.glob(os.path.join(ROOT, PKG, "csrc", "*")):
        for kind, target in inc.findall(open(p).read()):
            assert "oracle" not in target, (p, target)
    for p in glob.glob(os.path.join(ROOT, "oracle", "*.c")) + glob.glob(os.path.join(ROOT, "oracle", "*.h")):
        for kind, target in inc.findall(open(p).read()):
            assert kind == "<", (p, target)            # system headers only
            assert "zero" not in target, (p, target)
