"""Build the output-head shared library for sm_103a with nvcc.

Produces ``invariant_output_head_gb300/_lib/libdetlm_head.so`` in-tree (the
head's C ABI) and ``_lib/libdetlm_peak.so`` (the benchmark's dense-MMA rate
probe). One translation unit each, compiled in parallel, one ``-gencode``
(sm_103a); the CUDA runtime is linked statically so that the libraries load on
a machine without a GPU (for symbol checks) and use no libcuda symbol at link
time (the TMA descriptor encoder is fetched from the driver at run time).

Run as ``python -m invariant_output_head_gb300.build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc")
LIB_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIB_DIR, "libdetlm_head.so")
PEAK_LIB = os.path.join(LIB_DIR, "libdetlm_peak.so")
INCLUDE = os.path.join(ROOT, "include")
SOURCES = [os.path.join(SRC, "detlm_head.cu")]
TARGETS = {LIB: os.path.join(SRC, "detlm_head.cu"), PEAK_LIB: os.path.join(SRC, "mma_peak.cu")}
DEPS = SOURCES + [os.path.join(SRC, f) for f in os.listdir(SRC)] + \
    [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
         "-cudart", "static", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build")


def up_to_date() -> bool:
    for lib in TARGETS:
        if not os.path.exists(lib):
            return False
        t = os.path.getmtime(lib)
        if not all(os.path.getmtime(p) <= t for p in DEPS if os.path.exists(p)):
            return False
    return True


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(LIB_DIR, exist_ok=True)
    procs = []
    for lib, src in TARGETS.items():
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, *FLAGS, "-I", INCLUDE, "-I", SRC, "-o", tmp, src]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((lib, tmp, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                 stderr=subprocess.PIPE, text=True)))
    for lib, tmp, pr in procs:
        out, err = pr.communicate()
        if pr.returncode != 0:
            raise RuntimeError(f"nvcc failed ({pr.returncode}) for {lib}:\n{out}\n{err}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
