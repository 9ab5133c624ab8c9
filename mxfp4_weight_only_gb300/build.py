"""Build ``libmoe_a16w4.so`` in-tree for sm_103a with nvcc.

Each CUDA translation unit is compiled in parallel, then linked into one
shared library under ``mxfp4_weight_only_gb300/_build``.  The same sources
compiled with ``-DMOE_CHECK`` give the checked library
``libmoe_a16w4_check.so`` (kernels that bounds-check their indices into the
status word), built alongside.  Rebuilds only what is older than its sources.
Usage: ``python -m mxfp4_weight_only_gb300.build``.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB_NAME = "libmoe_a16w4.so"
CHECK_LIB_NAME = "libmoe_a16w4_check.so"
SOURCES = ["api.cu", "route.cu", "requant.cu", "decode.cu", "prefill.cu", "noalloc.cu", "actquant.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("common.cuh", "moe_internal.h")] + [
    os.path.join(ROOT, "include", "moe_a16w4.h")
]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_a16w4")


def lib_path(checked: bool = False) -> str:
    return os.path.join(BUILD, CHECK_LIB_NAME if checked else LIB_NAME)


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, jobs: int | None = None) -> str:
    """Build both libraries; returns the path of the regular one."""
    os.makedirs(os.path.join(BUILD, "check"), exist_ok=True)
    cc = nvcc()
    objs = {False: [], True: []}
    todo = []
    for checked in (False, True):
        for src in SOURCES:
            s = os.path.join(CSRC, src)
            o = os.path.join(BUILD, "check" if checked else "", src.replace(".cu", ".o"))
            objs[checked].append(o)
            if _stale(o, [s] + HEADERS):
                todo.append([cc] + FLAGS + (["-DMOE_CHECK"] if checked else []) + ["-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed ({r.returncode}) for {cmd[-3]}")

    with ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4) or 1) as ex:
        list(ex.map(run, todo))
    for checked in (False, True):
        lib = lib_path(checked)
        if todo or _stale(lib, objs[checked]):
            tmp = lib + ".tmp"
            run([cc] + ARCH + ["-shared", "-o", tmp] + objs[checked])
            os.replace(tmp, lib)
    return lib_path()


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
