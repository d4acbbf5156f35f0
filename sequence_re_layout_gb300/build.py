"""Compile the C-ABI library in-tree with nvcc for sm_103a: ``libbasp.so``
(release) and ``libbasp_debug.so`` (every kernel access bounds-checked)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libbasp.so")
DEBUG_LIB_PATH = os.path.join(PKG, "libbasp_debug.so")
SOURCES = ["layout.cpp", "relayout.cu"]
HEADERS = [os.path.join(INCLUDE, "basp.h"), os.path.join(INCLUDE, "basp_debug.h"),
           os.path.join(CSRC, "layout_internal.h"), os.path.join(CSRC, "relayout_kernel.cuh"),
           os.path.join(CSRC, "scratch_cache.h")]

NVCC_FLAGS = [
    "-O3", "-std=c++17",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo",
    "-Xcompiler", "-fPIC",
    "-shared",
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale(path) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS
    return any(os.path.getmtime(p) > t for p in deps)


def _command(out, extra, verbose):
    cmd = [_nvcc()] + NVCC_FLAGS + extra + ["-I", INCLUDE, "-o", out] + \
        [os.path.join(CSRC, s) for s in SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Build ``libbasp.so`` and ``libbasp_debug.so`` next to this file (the two
    in parallel) if missing or out of date; return the release library's path."""
    jobs = []
    for path, extra in ((LIB_PATH, []), (DEBUG_LIB_PATH, ["-DBASP_CHECK_BOUNDS=1"])):
        if force or _stale(path):
            tmp = path + ".tmp%d" % os.getpid()
            jobs.append((subprocess.Popen(_command(tmp, extra, verbose)), tmp, path))
    failed = False
    for proc, tmp, path in jobs:
        if proc.wait() != 0:
            failed = True
        elif not failed:
            os.replace(tmp, path)
    if failed:
        raise subprocess.CalledProcessError(1, "nvcc")
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
