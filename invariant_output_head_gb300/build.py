"""Build the output-head shared library for sm_103a with nvcc.

Produces ``invariant_output_head_gb300/_lib/libdetlm_head.so`` in-tree. One
translation unit, one ``-gencode`` (sm_103a); the CUDA runtime is linked
statically so that the library loads on a machine without a GPU (for symbol
checks) and uses no libcuda symbol at link time (the TMA descriptor encoder
is fetched from the driver at run time).

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
INCLUDE = os.path.join(ROOT, "include")
SOURCES = [os.path.join(SRC, "detlm_head.cu")]
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
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in DEPS if os.path.exists(p))


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, *FLAGS, "-I", INCLUDE, "-I", SRC, "-o", tmp, *SOURCES]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed ({r.returncode}):\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
