"""The CUDA path and the oracle are independent programs (CPU).

The library (`long_context_sparse_29_b300/`: the C ABI, its kernels, the
binding and its build) and the oracle (`oracle/`) share no code: neither
names, includes, imports or links the other.  Only the tests, the smoke run
and the benchmark's CPU legs (its `cpu_baseline` and its reference arm) call
the oracle; in `bench.py` it is imported inside those legs only, so the timed
GPU path never loads it.
"""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "long_context_sparse_29_b300")
ORC = os.path.join(ROOT, "oracle")


def _sources(top, exts):
    for dp, dn, fn in os.walk(top):
        dn[:] = [d for d in dn if d not in ("_build", "__pycache__")]
        for f in fn:
            if f.endswith(exts):
                yield os.path.join(dp, f)


def test_library_never_names_the_oracle():
    files = list(_sources(PKG, (".py", ".cu", ".cuh", ".h", ".c")))
    assert len(files) >= 10
    for p in files:
        with open(p, encoding="utf-8") as f:
            assert "oracle" not in f.read().lower(), p


def test_oracle_never_names_the_library():
    files = list(_sources(ORC, (".py", ".c", ".h")))
    assert len(files) >= 2
    for p in files:
        with open(p, encoding="utf-8") as f:
            text = f.read()
        for name in ("long_context_sparse_29_b300", "libcsa_b300", "csrc", "csa_common", "attn_common",
                     "tc_ptx", "launch.h"):
            assert name not in text, (p, name)


def test_bench_imports_the_oracle_only_in_its_cpu_legs():
    with open(os.path.join(ROOT, "bench.py"), encoding="utf-8") as f:
        tree = ast.parse(f.read())
    found = []

    def walk(node, where):
        for ch in ast.iter_child_nodes(node):
            w = ch.name if isinstance(ch, (ast.FunctionDef, ast.AsyncFunctionDef)) else where
            if isinstance(ch, (ast.Import, ast.ImportFrom)):
                names = [a.name for a in ch.names]
                if isinstance(ch, ast.ImportFrom) and ch.module:
                    names.append(ch.module)
                if any(n.split(".")[0] == "oracle" for n in names):
                    found.append(w)
            walk(ch, w)

    walk(tree, None)
    assert found and set(found) <= {"oracle_sample", "cpu_baseline", "run_reference"}, found
