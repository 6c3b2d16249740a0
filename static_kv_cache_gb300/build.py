"""Build libkvc.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

The decode kernels are compiled once per (element type, head width) from
``kvc_decode_inst.cu`` so that the translation units build in parallel.
Objects go to ``_build/`` at the repository root; the library lands next to
this file, where the Python binding loads it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", "kvc")
LIB = os.path.join(PKG, "libkvc.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]

ELEM_TYPES = {"bf16": 0, "f16": 1, "f32": 2}
HEAD_DIMS = (32, 64, 128, 256)


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libkvc.so")


def _units():
    units = []
    for src in ("kvc_api.cu", "kvc_append.cu", "kvc_noalloc.cu", "kvc_mla_api.cu"):
        units.append((os.path.join(CSRC, src), os.path.join(BUILD, src.replace(".cu", ".o")), []))
    inst = os.path.join(CSRC, "kvc_decode_inst.cu")
    for tag, code in ELEM_TYPES.items():
        for d in HEAD_DIMS:
            obj = os.path.join(BUILD, f"kvc_decode_{tag}_{d}.o")
            units.append((inst, obj, [f"-DKVC_INST_TYPE={code}", f"-DKVC_INST_D={d}"]))
    for tag, code in (("bf16", 0), ("f16", 1)):
        for d in (64, 128):
            units.append((inst, os.path.join(BUILD, f"kvc_decode_paged_{tag}_{d}.o"),
                          [f"-DKVC_INST_TYPE={code}", f"-DKVC_INST_D={d}", "-DKVC_INST_PAGED"]))
        units.append((inst, os.path.join(BUILD, f"kvc_decode_tc_{tag}_128.o"),
                      [f"-DKVC_INST_TYPE={code}", "-DKVC_INST_D=128", "-DKVC_INST_TC"]))
    units.append((os.path.join(CSRC, "kvc_decode_q8_inst.cu"), os.path.join(BUILD, "kvc_decode_q8_128.o"), []))
    pre = os.path.join(CSRC, "kvc_prefill_inst.cu")
    for code, tag in ((0, "bf16"), (1, "f16")):
        for d in (64, 128):
            obj = os.path.join(BUILD, f"kvc_prefill_{tag}_{d}.o")
            units.append((pre, obj, [f"-DKVC_INST_TYPE={code}", f"-DKVC_INST_D={d}"]))
    mla = os.path.join(CSRC, "kvc_mla_inst.cu")
    for code, tag in ((0, "bf16"), (1, "f16")):
        units.append((mla, os.path.join(BUILD, f"kvc_mla_{tag}.o"), [f"-DKVC_INST_TYPE={code}"]))
    return units


def _deps():
    return (glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(unit, extra_flags, verbose):
    src, obj, defs = unit
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra_flags, *defs, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(obj)}:\n{r.stderr}")
    return r.stderr if verbose else ""


def build(force: bool = False, jobs: int | None = None, extra_flags=(), verbose: bool = False) -> str:
    """Compile every kernel unit and link libkvc.so; returns its path."""
    deps = _deps()
    if not force and not _stale(LIB, deps):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    units = _units()
    todo = [u for u in units if force or _stale(u[1], deps)]
    jobs = jobs or min(len(todo) or 1, max(2, os.cpu_count() or 2))
    logs = []
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        for out in ex.map(lambda u: _compile(u, list(extra_flags), verbose), todo):
            logs.append(out)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[u[1] for u in units]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print("".join(logs))
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
