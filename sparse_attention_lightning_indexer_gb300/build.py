"""Builds the ds4idx shared library in-tree (nvcc, sm_103a only).

Output: ``sparse_attention_lightning_indexer_gb300/_lib/libds4idx.so``. Every ``csrc/*.cu`` file
is compiled to an object in parallel, then the objects are linked into one library. The CUDA
runtime is linked statically; the driver's tensor-map encoder is resolved at run time, so the
library needs no libcuda at link time and cross-compiles on a machine without a GPU.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libds4idx.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC"]
LINK_FLAGS = [*ARCH, "-shared", "--cudart", "static"]


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def deps() -> list[str]:
    """Every file the library is compiled from: the sources, all csrc headers, the C header."""
    headers = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                     if f.endswith((".cuh", ".h", ".cu")))
    return sorted(set(sources() + headers + [os.path.join(INCLUDE, f)
                                             for f in os.listdir(INCLUDE) if f.endswith(".h")]))


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    tag = f".tmp{os.getpid()}"
    objs, procs = [], []
    for src in sources():
        obj = os.path.join(LIB_DIR, os.path.basename(src)[:-3] + tag + ".o")
        cmd = [nvcc(), *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((subprocess.Popen(cmd), cmd))
        objs.append(obj)
    failed = [cmd for p, cmd in procs if p.wait() != 0]
    try:
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        tmp = LIB_PATH + tag
        cmd = [nvcc(), *LINK_FLAGS, *objs, "-o", tmp]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB_PATH)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
