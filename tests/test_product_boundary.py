"""The product path and the oracle stay apart: no module of the package
imports the oracle (there is no CPU fallback), the oracle imports nothing of
the package, and the binding fails loudly when the CUDA library is absent."""
import ast
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "block_fp8_mixture_route_gb300")


def imported_modules(path):
    tree = ast.parse(open(path).read())
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom):
            yield ("." * node.level) + (node.module or "")


def test_package_never_imports_the_oracle():
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith(".py"):
                mods = list(imported_modules(os.path.join(dirpath, f)))
                assert not any(m == "oracle" or m.startswith("oracle.") for m in mods), (f, mods)
    for dirpath, _, files in os.walk(os.path.join(PKG, "csrc")):
        for f in files:
            assert "oracle" not in open(os.path.join(dirpath, f), errors="ignore").read().lower(), f


def test_oracle_imports_nothing_of_the_package():
    odir = os.path.join(ROOT, "oracle")
    for f in os.listdir(odir):
        if f.endswith(".py"):
            mods = list(imported_modules(os.path.join(odir, f)))
            assert not any("block_fp8_mixture_route_gb300" in m for m in mods), (f, mods)


def test_missing_library_fails_loudly():
    code = ("from block_fp8_mixture_route_gb300 import _lib\n"
            "try:\n    _lib.load('/nonexistent/libmoe_fp8_block.so')\n"
            "except RuntimeError as e:\n    print('raised:', e)\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, timeout=300)
    assert r.returncode == 0 and "raised: CUDA library not built" in r.stdout, r.stdout + r.stderr
