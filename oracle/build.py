"""Compile the C oracle (``kvc_oracle.c``) into ``oracle/_build/libkvc_oracle.so``.

TEST INFRASTRUCTURE ONLY: the oracle is the checker, never the product path.

Plain ``gcc``: ``-O2`` without fast-math and with ``-ffp-contract=off`` so
that x86_64 and aarch64 hosts evaluate the same fp64 expression tree.  OpenMP
(parallel over (sequence, query head), nothing else) is used when the
compiler supports it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kvc_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libkvc_oracle.so")

BASE_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
              "-fno-fast-math", "-Wall"]


def compile_source(src: str, out: str, openmp: bool = True) -> str:
    """Compile one oracle source file to a shared library at ``out``."""
    cc = os.environ.get("CC", "gcc")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [cc, *BASE_FLAGS, src, "-o", tmp, "-lm"]
    if openmp:
        try:
            subprocess.run(cmd[:1] + ["-fopenmp"] + cmd[1:], check=True,
                           capture_output=True, text=True)
        except subprocess.CalledProcessError:
            subprocess.run(cmd, check=True, capture_output=True, text=True)
    else:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    return compile_source(SRC, LIB)


def build_variant(source_text: str, tag: str) -> str:
    """Compile a modified copy of the oracle source (used by the tests that
    plant a mistake in the oracle and check that a pin catches it)."""
    d = tempfile.mkdtemp(prefix=f"kvo_{tag}_")
    src = os.path.join(d, "kvc_oracle_variant.c")
    with open(src, "w") as f:
        f.write(source_text)
    out = os.path.join(d, "libkvc_oracle_variant.so")
    try:
        return compile_source(src, out, openmp=False)
    except subprocess.CalledProcessError:
        shutil.rmtree(d, ignore_errors=True)
        raise


if __name__ == "__main__":
    print(build(force=True))
