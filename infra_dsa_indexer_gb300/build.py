"""Build the C-ABI CUDA library in-tree: infra_dsa_indexer_gb300/_build/libdsa_indexer.so.

One translation unit, one -gencode (sm_103a), compiled with nvcc; no cmake.
Run `python -m infra_dsa_indexer_gb300.build` or call build().
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libdsa_indexer.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
SOURCES = ["indexer_api.cu"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "dsa_indexer.h"))
    files.append(os.path.abspath(__file__))
    return files


def nvcc_command(out_path: str, extra=()):
    nvcc = os.environ.get("NVCC", "nvcc")
    return [nvcc, *ARCH_FLAGS, "-O3", "-std=c++17", "-lineinfo", "-shared",
            "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
            "-I", INCLUDE, "-I", CSRC, *extra, "-o", out_path,
            *[os.path.join(CSRC, s) for s in SOURCES]]


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile the library if any source is newer than it; return its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(LIB_PATH):
        lib_t = os.path.getmtime(LIB_PATH)
        if all(os.path.getmtime(f) <= lib_t for f in _inputs()):
            return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = nvcc_command(tmp, extra)
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.check_call(cmd)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ()))
