"""The CUDA path and the oracle share no code, and the product has no CPU
fallback (CPU only, no GPU needed):

- no module of the package imports ``oracle`` and no CUDA source includes an
  oracle header or names its sources; the oracle in turn neither imports the
  package nor includes a CUDA-side header;
- ``bench.py`` reaches the oracle only inside its CPU-baseline and reference
  legs, and ``__graft_entry__`` only inside ``build()`` (compiling the checker)
  and ``smoke()`` (checking against it);
- the seeded input generators (``workloads.py``) import neither side;
- importing the package when ``libmoe_ep.so`` is missing raises instead of
  running anything else.
"""
import ast
import glob
import importlib.util
import os
import re
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG_NAME = "combine_moe_dispatch_layout_gb300"
PKG = os.path.join(ROOT, PKG_NAME)


def _imports(path):
    """(module name, enclosing top-level function or None) of every import."""
    tree = ast.parse(open(path).read(), filename=path)
    out = []

    def walk(node, func):
        for child in ast.iter_child_nodes(node):
            f = func
            if func is None and isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef,
                                                   ast.ClassDef)):
                f = child.name
            if isinstance(child, ast.Import):
                out.extend((a.name, f) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                mod = child.module or ""
                if child.level:
                    mod = "." * child.level + mod
                out.append((mod, f))
            walk(child, f)

    walk(tree, None)
    return out


def _top(mod):
    return mod.lstrip(".").split(".")[0]


def test_package_never_imports_the_oracle():
    files = glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True)
    assert files
    for path in files:
        for mod, _ in _imports(path):
            assert _top(mod) not in ("oracle", "workloads", "tests"), (path, mod)


def test_cuda_sources_share_nothing_with_the_oracle():
    srcs = glob.glob(os.path.join(PKG, "csrc", "*"))
    assert any(s.endswith(".cu") for s in srcs)
    oracle_files = {os.path.basename(p) for p in glob.glob(os.path.join(ROOT, "oracle", "*"))
                    if p.endswith((".c", ".h"))}
    assert oracle_files
    for path in srcs:
        text = open(path).read()
        for inc in re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', text):
            assert os.path.basename(inc) not in oracle_files, (path, inc)
            assert "oracle" not in inc, (path, inc)
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.[ch]")):
        text = open(path).read()
        for inc in re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', text):
            assert not inc.startswith("moe_ep"), (path, inc)
            assert not inc.endswith(".cuh"), (path, inc)


def test_oracle_never_imports_the_package():
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        for mod, _ in _imports(path):
            assert _top(mod) not in (PKG_NAME, "workloads", "bench"), (path, mod)


def test_input_generators_import_neither_side():
    for mod, _ in _imports(os.path.join(ROOT, "workloads.py")):
        assert _top(mod) not in (PKG_NAME, "oracle"), mod


def test_bench_reaches_the_oracle_only_in_its_cpu_legs():
    path = os.path.join(ROOT, "bench.py")
    users = {f for mod, f in _imports(path) if _top(mod) == "oracle"}
    assert users and users <= {"cpu_baseline", "run_reference", "OracleHost"}, users
    # and the class that runs the oracle is used only by those two legs
    tree = ast.parse(open(path).read(), filename=path)
    for top in tree.body:
        if isinstance(top, (ast.FunctionDef, ast.ClassDef)) and top.name not in (
                "cpu_baseline", "run_reference", "OracleHost"):
            names = {n.id for n in ast.walk(top) if isinstance(n, ast.Name)}
            assert "OracleHost" not in names, top.name


def test_entry_reaches_the_oracle_only_in_build_and_smoke():
    users = {f for mod, f in _imports(os.path.join(ROOT, "__graft_entry__.py"))
             if _top(mod) == "oracle"}
    assert users and users <= {"build", "smoke"}, users


def test_import_without_the_library_raises(tmp_path):
    """A copy of the package with no libmoe_ep.so beside it refuses to import."""
    dst = tmp_path / PKG_NAME
    dst.mkdir()
    for path in glob.glob(os.path.join(PKG, "*.py")):
        shutil.copy(path, dst / os.path.basename(path))
    assert not (dst / "libmoe_ep.so").exists()
    name = "_moe_ep_without_library"
    spec = importlib.util.spec_from_file_location(name, str(dst / "__init__.py"),
                                                  submodule_search_locations=[str(dst)])
    module = importlib.util.module_from_spec(spec)
    sys.modules[name] = module
    try:
        with pytest.raises(ImportError, match="not built"):
            spec.loader.exec_module(module)
    finally:
        sys.modules.pop(name, None)
