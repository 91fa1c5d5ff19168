"""Builds the C-ABI library ``lib/libfa.so`` from ``csrc/`` with nvcc for sm_103a.

The library is one translation unit (``csrc/fa_lib.cu``) with the CUDA runtime
linked statically, so it loads with ``ctypes`` on any host and depends on no
particular torch build.  Rebuilds only when a source is newer than the output.
"""

from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
CSRC_DIR = os.path.join(PKG_DIR, "csrc")
INCLUDE_DIR = os.path.join(REPO_DIR, "include")
LIB_DIR = os.path.join(PKG_DIR, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libfa.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")


def _sources():
    srcs = [os.path.join(CSRC_DIR, f) for f in sorted(os.listdir(CSRC_DIR)) if f.endswith((".cu", ".cuh"))]
    srcs.append(os.path.join(INCLUDE_DIR, "fa.h"))
    return srcs


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    out_t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(s) > out_t for s in _sources())


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile libfa.so if needed and return its path."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIB_PATH + ".tmp"
    cmd = [_nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", INCLUDE_DIR, "-o", tmp, os.path.join(CSRC_DIR, "fa_lib.cu")]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd))
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
