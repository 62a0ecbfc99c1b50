"""The oracle is test infrastructure and the CUDA path does not use it.

Static checks on the sources: nothing in the package imports, loads or names
the oracle; the oracle does not import the package, include its CUDA sources
or load libdtrot; and the two share no source file.  Only the seeded input
generators (workloads.py, which holds none of the method's arithmetic) serve
both sides.
"""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "diffusion_transformer_elementwise_rotate_b300")
ORACLE = os.path.join(ROOT, "oracle")


def _sources(d, exts):
    out = []
    for ext in exts:
        out += glob.glob(os.path.join(d, "**", "*" + ext), recursive=True)
    return [p for p in out if "__pycache__" not in p and "_build" not in p]


def test_package_never_touches_the_oracle():
    pat = re.compile(r"\boracle\b|liboracle|dtrot_oracle|dto_")
    for p in _sources(PKG, (".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
        text = open(p, encoding="utf-8").read()
        hits = [l for l in text.splitlines() if pat.search(l)]
        assert not hits, f"{os.path.relpath(p, ROOT)} mentions the oracle: {hits[:3]}"


def test_oracle_never_touches_the_cuda_path():
    pat = re.compile(r"diffusion_transformer_elementwise_rotate_b300|libdtrot|dtrot\.h|"
                     r"dtrot_internal|csrc/|\.cu\b|_capi")
    for p in _sources(ORACLE, (".py", ".c", ".h")):
        text = open(p, encoding="utf-8").read()
        code = [l for l in text.splitlines()
                if pat.search(l) and not l.lstrip().startswith(("#", "*", "//", "/*"))]
        assert not code, f"{os.path.relpath(p, ROOT)} reaches into the CUDA path: {code[:3]}"


def test_no_shared_source_files():
    pkg = {os.path.basename(p) for p in _sources(PKG, (".py", ".cu", ".cuh", ".c", ".h"))}
    orc = {os.path.basename(p) for p in _sources(ORACLE, (".py", ".c", ".h"))}
    assert pkg & orc <= {"__init__.py", "build.py"}, pkg & orc


def test_oracle_headers_say_it_is_test_infrastructure():
    for name in ("__init__.py", "dtrot_oracle.c"):
        head = open(os.path.join(ORACLE, name), encoding="utf-8").read()[:2000].lower()
        assert "test infrastructure" in head or "only the tests" in head, name
