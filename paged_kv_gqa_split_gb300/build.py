"""Build the sm_103a shared library in-tree with nvcc (no cmake, no torch extension).

``python -m paged_kv_gqa_split_gb300.build`` (or ``build()``) compiles the CUDA
translation units in parallel and links ``libgqa_paged_decode.so`` next to this
file. Objects go to ``_build/`` inside the package; both are git-ignored.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from typing import List

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libgqa_paged_decode.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
SOURCES = ["gqa_decode_lsu.cu", "gqa_decode_tma.cu", "gqa_merge.cu", "gqa_api.cu", "gqa_noalloc.cu", "gqa_kv_append.cu",
           "gqa_sparse.cu", "gqa_mla.cu", "gqa_mla_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    for p in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(p):
            return p
    raise RuntimeError("nvcc not found; the CUDA toolkit (13.x) is required to build the library")


def _flags(extra: List[str]) -> List[str]:
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O3", "-I", INCLUDE, "-I", CSRC] + extra


def _run(cmd: List[str], verbose: bool) -> str:
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"command failed ({res.returncode}): {' '.join(cmd)}\n{res.stdout}")
    return res.stdout


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    lib_t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    deps.append(os.path.abspath(__file__))  # the source list lives here
    return any(os.path.getmtime(d) > lib_t for d in deps)


def build(verbose: bool = False, force: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile and link the library if any source is newer than it. Returns its path."""
    if not force and not _stale():
        return LIB_PATH
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        out = _run([nvcc] + _flags(extra) + ["-c", os.path.join(CSRC, src), "-o", obj], verbose)
        if ptxas_verbose:
            print(out)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + ".tmp"
    _run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs, verbose)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    path = build(verbose=True, force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv)
    print(path)
