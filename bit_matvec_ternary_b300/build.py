"""Build libtl.so (the C-ABI library) in-tree for sm_103a with nvcc.

    python -m bit_matvec_ternary_b300.build [--force] [--verbose]

The library links the CUDA runtime statically, so loading it needs no
particular libcudart on the library path; it does not link the driver library
either (the driver is reached through the runtime), so it loads on machines
without a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libtl.so")
BUILD_DIR = os.path.join(PKG, "_build")

SOURCES = ["tl_host.cpp", "tl_kernels.cu", "tl_prefill.cu", "tl_head.cu", "tl_fused.cu", "tl_blockscale.cu", "tl_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "tl.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    objs = []
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-Xcompiler", "-fPIC,-fvisibility=hidden"]
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src + ".o")
        cmd = [nvcc()] + common + ARCH + ["-lineinfo", "-c", path, "-o", obj]
        if src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"] if verbose else []
        else:
            cmd += ["-x", "c++"]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.check_call(cmd)
        objs.append(obj)
    tmp = LIB + ".tmp"
    link = [nvcc(), "-shared", "-cudart", "static"] + ARCH + objs + ["-o", tmp]
    if verbose:
        print(" ".join(link), flush=True)
    subprocess.check_call(link)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
