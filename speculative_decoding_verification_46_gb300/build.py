"""Compile libspecverify.so in-tree for sm_103a with nvcc.

    python -m speculative_decoding_verification_46_gb300.build [--force]

The output goes to ``speculative_decoding_verification_46_gb300/lib/`` (git
ignored).  The library is rebuilt when a source or header is newer than it.
"""

from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIBNAME = "libspecverify.so"
LIB_PATH = os.path.join(LIBDIR, LIBNAME)

SOURCES = ["sv_api.cu", "sv_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Build (if stale) and return the path of libspecverify.so."""
    if not force and os.path.exists(LIB_PATH):
        lib_mtime = os.path.getmtime(LIB_PATH)
        if all(os.path.getmtime(f) <= lib_mtime for f in _inputs()):
            return LIB_PATH
    os.makedirs(LIBDIR, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           f"-I{INCLUDE}", "-o", tmp, *[os.path.join(CSRC, s) for s in SOURCES]]
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True))
