"""The product path and the oracle, checked on the CPU by reading the sources:
they share no code and neither imports or includes the other; outside
tests/, the oracle is touched only by __graft_entry__ (build compiles it,
smoke checks against it) and by bench.py's CPU-baseline and reference legs;
and the binding raises on import when the CUDA library is missing, so there
is no silent fallback."""
import ast
import os
import re
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "block_scaled_fp8_router_gb300")
ORACLE = os.path.join(ROOT, "oracle")
SKIP_DIRS = {"__pycache__", "lib", "_build"}


def _sources(top, exts):
    for dp, dns, fns in os.walk(top):
        dns[:] = [d for d in dns if d not in SKIP_DIRS]
        for fn in fns:
            if fn.endswith(exts):
                yield os.path.join(dp, fn)


def _imports(tree):
    """(module name, enclosing function names) of every import in a module."""
    out = []

    def walk(node, stack):
        for child in ast.iter_child_nodes(node):
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef, ast.ClassDef)):
                walk(child, stack + [child.name])
                continue
            if isinstance(child, ast.Import):
                out.extend((a.name, tuple(stack)) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                out.append((child.module or "", tuple(stack)))
            walk(child, stack)

    walk(tree, [])
    return out


def _is_oracle(mod):
    return mod == "oracle" or mod.startswith("oracle.")


def _includes(path):
    return re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', open(path).read())


def test_package_never_touches_the_oracle():
    for path in _sources(PKG, (".py",)):
        src = open(path).read()
        assert not any(_is_oracle(m) for m, _ in _imports(ast.parse(src))), path
        assert "liboracle" not in src and "moe_oracle" not in src, path
    for path in _sources(PKG, (".cu", ".cuh", ".h", ".c", ".cpp")):
        assert not any("oracle" in inc for inc in _includes(path)), path


def test_oracle_never_touches_the_package():
    for path in _sources(ORACLE, (".c", ".h")):
        # the C oracle includes only the C library (and OpenMP): no CUDA header, no csrc header, no moe_r3.h
        assert all(inc in ("math.h", "stdint.h", "stdlib.h", "string.h", "omp.h") for inc in _includes(path)), path
    for path in _sources(ORACLE, (".py",)):
        src = open(path).read()
        for mod, _ in _imports(ast.parse(src)):
            assert not mod.startswith("block_scaled_fp8_router_gb300") and mod not in ("torch", "bench"), (path, mod)
        assert "libmoe_r3" not in src and "csrc" not in src, path


def test_oracle_users_outside_the_tests():
    """bench.py imports the oracle only in its CPU legs (the oracle sample,
    the CPU baseline, and main's reference arm); __graft_entry__ only in
    build and smoke."""
    allowed = {
        "bench.py": {("OracleSample", "__init__"), ("OracleSample", "_ids"), ("OracleSample", "run"),
                     ("cpu_baseline",), ("cpu_config_legs",), ("main",)},
        "__graft_entry__.py": {("build",), ("smoke",)},
    }
    for name, ok in allowed.items():
        tree = ast.parse(open(os.path.join(ROOT, name)).read())
        users = {where for mod, where in _imports(tree) if _is_oracle(mod)}
        assert users and users <= ok, (name, users - ok)
    # in main, only the reference arm's branch imports it
    main = next(n for n in ast.parse(open(os.path.join(ROOT, "bench.py")).read()).body
                if isinstance(n, ast.FunctionDef) and n.name == "main")
    for node in ast.walk(main):
        if isinstance(node, ast.If) and "reference" in ast.unparse(node.test):
            ref_branch = {id(n) for n in ast.walk(node)}
            break
    else:
        raise AssertionError("main has no reference branch")
    for node in ast.walk(main):
        if isinstance(node, (ast.Import, ast.ImportFrom)):
            mods = [a.name for a in node.names] if isinstance(node, ast.Import) else [node.module or ""]
            if any(_is_oracle(m) for m in mods):
                assert id(node) in ref_branch, ast.unparse(node)


def test_binding_raises_without_the_library(tmp_path):
    """A copy of the package without its built library cannot be imported:
    neither the binding nor the layer falls back to anything."""
    dst = tmp_path / "block_scaled_fp8_router_gb300"
    dst.mkdir()
    for fn in os.listdir(PKG):
        if fn.endswith(".py"):
            shutil.copy(os.path.join(PKG, fn), dst / fn)
    for mod in ("moe_r3", "layer"):
        code = (f"import sys; sys.path.insert(0, {str(tmp_path)!r})\n"
                f"try:\n    import block_scaled_fp8_router_gb300.{mod}\nexcept ImportError as e:\n"
                f"    print('raised:', e)\nelse:\n    print('imported')\n")
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, cwd=tmp_path)
        assert r.returncode == 0, r.stderr[-2000:]
        assert r.stdout.startswith("raised:") and "libmoe_r3.so is not built" in r.stdout, r.stdout
