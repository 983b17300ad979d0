"""Build libmagicpig.so in-tree from csrc/*.cu with nvcc for sm_103a.

Usage: python lsh_sampled_sparse_centered_gb300/build.py [-v] [-f] [--check]   (run by path:
the package itself cannot be imported before the library exists), or
__graft_entry__.build(). The translation units compile in parallel; the shared library
links the CUDA runtime dynamically with an rpath to the toolkit's lib64. --check builds
the bounds-checking library libmagicpig_check.so (MP_CHECK=1: kernels test every index
that comes from data before using it and report failures in the status word), which the
binding loads instead when MP_BOUNDS_CHECK=1 is set.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libmagicpig.so")
LIB_CHECK = os.path.join(OUT_DIR, "libmagicpig_check.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_lib64(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(verbose: bool = False, force: bool = False, check: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    srcs = sources()
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(ROOT, "include", "magicpig.h"))
    lib = LIB_CHECK if check else LIB
    if not force and os.path.exists(lib):
        t = os.path.getmtime(lib)
        if all(os.path.getmtime(d) <= t for d in deps):
            return lib
    flags = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
             "-I" + os.path.join(ROOT, "include"), "-I" + CSRC] + ARCH + (["-DMP_CHECK=1"] if check else [])
    objs = []

    def compile_one(src: str) -> str:
        obj = os.path.join(OUT_DIR, os.path.basename(src)[:-3] + ("_check" if check else "") + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc, "-shared", "-cudart", "shared", "-o", tmp] + objs + ARCH + [
        "-Xlinker", "-rpath," + _cuda_lib64(nvcc)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, check="--check" in sys.argv))
