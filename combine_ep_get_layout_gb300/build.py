"""Builds ``libep_gb300.so`` (the C-ABI library) from ``csrc/`` with nvcc.

    python -m combine_ep_get_layout_gb300.build [--force] [--verbose] [--trace]

One ``-gencode arch=compute_103a,code=sm_103a`` target, translation units
compiled in parallel, objects under ``_build/`` beside this file, the shared
library beside this file.  Nothing is installed anywhere else.

``--trace`` builds ``libep_gb300_trace.so`` instead: the same sources with
``EP_TRACE`` defined, so the kernels record per-block timeline marks (see
``csrc/ep_trace.cuh`` and ``trace.py``).  The product library never has them.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libep_gb300.so")

SOURCES = ["ep_api.cu", "ep_layout.cu", "ep_layout_expanded.cu", "ep_dispatch.cu", "ep_combine.cu",
           "ep_noalloc.cu", "ep_selftest.cu"]
HEADERS = ["ep_device.cuh", "ep_internal.h", "ep_trace.cuh"]
TRACE_LIB = os.path.join(HERE, "libep_gb300_trace.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
         "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or install the CUDA toolkit)")


def _inputs() -> list[str]:
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS]
            + [os.path.join(INCLUDE, "ep_gb300.h"), os.path.abspath(__file__)])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, trace: bool = False) -> str:
    """Compile the library (or with ``trace`` the trace build) if a source
    is newer than it; return its path."""
    lib = TRACE_LIB if trace else LIB
    if not force and up_to_date(lib):
        return lib
    build_dir = os.path.join(BUILD, "trace") if trace else BUILD
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if trace:
        extra.append("-DEP_TRACE")

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(p.stdout + p.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, lib)
    return lib


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print registers / spills / smem")
    ap.add_argument("--trace", action="store_true", help="the trace build (per-block timeline marks)")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, ptxas_info=a.ptxas_info, trace=a.trace))
    return 0


if __name__ == "__main__":
    sys.exit(main())
