"""Builds the CUDA library libmtl.so in-tree for sm_103a with nvcc.

Each translation unit under csrc/ compiles in parallel to an object file, then
one link step makes the shared library.  Run as a script or call build().
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmtl.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libmtl_debug.so")
ROOT = os.path.dirname(PKG)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src: str, verbose_ptxas: bool, debug: bool = False) -> str:
    obj = os.path.join(BUILD_DEBUG if debug else BUILD, os.path.basename(src)[:-3] + ".o")
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(ROOT, "include", "mtl.h"))
    if (not verbose_ptxas and os.path.exists(obj)
            and os.path.getmtime(obj) >= max(os.path.getmtime(d) for d in deps)):
        return obj
    cmd = [nvcc(), *ARCH, *FLAGS, *(["-DMTL_DEBUG"] if debug else []), "-c", src, "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def build(verbose_ptxas: bool = False, debug: bool = False) -> str:
    """Builds libmtl.so, or with debug the MTL_DEBUG build libmtl_debug.so
    (device-side checks of computed TMA coordinates and output indices that
    report MTL_ERR_BOUNDS instead of faulting).  Returns the library's path."""
    out_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(out_dir, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, debug), srcs))
    if (not os.path.exists(lib)
            or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs)):
        tmp = lib + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
