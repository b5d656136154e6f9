"""Build ``libmaxsim.so`` in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel to ``_build/*.o``; the objects
link into one shared library with the CUDA runtime linked statically, so the
library loads on a machine without a GPU driver (nothing runs until a call).
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
SOURCES = ["maxsim_api.cu", "fwd_tc.cu", "bwd.cu", "noalloc.cu", "topk.cu", "chamfer.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def library_path() -> str:
    return os.path.join(PKG, "libmaxsim.so")


def _nvcc() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found")
    return nvcc


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "maxsim.h"))
    return files


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    out = library_path()
    if not force and os.path.exists(out):
        newest = max(os.path.getmtime(f) for f in _deps())
        if os.path.getmtime(out) >= newest:
            return out
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    flags = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose_ptxas:
        for _, log in results:
            print(log)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", *ARCH, "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
