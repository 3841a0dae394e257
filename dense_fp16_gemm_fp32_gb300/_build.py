"""Builds the CUDA library ``libgemm_sm103.so`` in-tree with nvcc (sm_103a only).

One translation unit per API file (csrc/gemm_api.cu with the GEMM kernels,
csrc/softmax_api.cu with the softmax kernels), compiled in parallel with one
-gencode each and linked into one shared library, so a build takes seconds.
The shared cudart is used so the library and PyTorch share one CUDA runtime
in the process.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libgemm_sm103.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
UNITS = ["gemm_api.cu", "softmax_api.cu"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libgemm_sm103.so")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    """Compile the library if it is missing or older than a source file."""
    if not force and not stale():
        return LIB
    nvcc = _nvcc()
    tag = f".tmp{os.getpid()}"
    tmp = LIB + tag
    compile_flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{INCLUDE}",
                     *(extra_flags or [])]
    objs, procs = [], []
    for unit in UNITS:
        obj = os.path.join(PKG, f"{os.path.splitext(unit)[0]}.{os.getpid()}.o")
        cmd = [nvcc, *compile_flags, "-c", "-o", obj, os.path.join(CSRC, unit)]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        objs.append(obj)
        procs.append(subprocess.Popen(cmd))
    try:
        failed = [p.args[-1] for p in procs if p.wait() != 0]
        if failed:
            raise subprocess.CalledProcessError(1, f"nvcc {' '.join(failed)}")
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", f"-rpath,{_cuda_lib_dir(nvcc)}",
               "-o", tmp, *objs]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None))
