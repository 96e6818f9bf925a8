"""The oracle and the GPU path share no code, and the product never runs the
oracle: checked on the sources.

- Nothing in the package (Python binding, CUDA sources, C ABI header) imports,
  includes or loads anything from ``oracle/``.
- Nothing in ``oracle/`` imports or includes anything from the package or the
  header; the oracle's C file includes only C standard and POSIX headers.
- Only the test suite, ``__graft_entry__`` (build and smoke) and ``bench.py``
  (its CPU baseline and reference legs) name the oracle.
"""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "dense_matmul_tensor_gb300")


def _sources(top, exts):
    for d, _, files in os.walk(top):
        if "_lib" in d or "__pycache__" in d:
            continue
        for f in files:
            if f.endswith(exts):
                yield os.path.join(d, f)


def test_package_never_uses_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#\s*include\s*[<\"][^>\"]*oracle)|liboracle", re.M)
    for path in list(_sources(PKG, (".py", ".cu", ".cuh", ".h", ".c"))) + [os.path.join(ROOT, "include", "bmm.h")]:
        text = open(path, encoding="utf-8").read()
        assert not pat.search(text), f"{path} refers to the oracle"


def test_oracle_never_uses_the_package():
    pat = re.compile(r"dense_matmul_tensor_gb300|bmm\.h|libdmt_bmm|csrc")
    for path in _sources(os.path.join(ROOT, "oracle"), (".py", ".c", ".h")):
        text = open(path, encoding="utf-8").read()
        code = "\n".join(l for l in text.splitlines() if not l.lstrip().startswith(("#", "*", "//", "/*")) or
                         l.lstrip().startswith("#include"))
        assert not pat.search(code), f"{path} refers to the GPU package"
    includes = re.findall(r"#\s*include\s*[<\"]([^>\"]+)", open(os.path.join(ROOT, "oracle", "bmm_oracle.c")).read())
    assert set(includes) <= {"math.h", "pthread.h", "stdint.h", "stdlib.h", "string.h", "stdio.h"}, includes


def test_only_tests_entry_and_bench_name_the_oracle():
    allowed = {os.path.join(ROOT, "__graft_entry__.py"), os.path.join(ROOT, "bench.py")}
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle\s+import)", re.M)
    for path in _sources(ROOT, (".py",)):
        rel = os.path.relpath(path, ROOT)
        if rel.startswith(("tests" + os.sep, "oracle" + os.sep, "_work" + os.sep, "baseline" + os.sep)):
            continue
        if pat.search(open(path, encoding="utf-8").read()):
            assert path in allowed, f"{rel} imports the oracle"
