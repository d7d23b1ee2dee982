"""Builds libtb.so (the CUDA library) in-tree with nvcc for sm_103a.

Each .cu file under csrc/ is compiled in parallel to an object file under
_build/, then linked into ln_backward_gb300/libtb.so against the shared CUDA
runtime.  No cmake, one -gencode.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libtb.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtb.so")


def cuda_home(nvcc: str) -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def cflags(extra=()):
    return ["-std=c++17", "-O3", ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O2",
            "-Xptxas", "-O3", f"-I{INCLUDE}", f"-I{CSRC}", *extra]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, ptxas_verbose: bool = False) -> str:
    nvcc = nvcc_path()
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "tb.h"))
    srcs = sources()
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []

    def compile_one(src_obj):
        src, obj = src_obj
        if not force and not ptxas_verbose and not _stale(obj, [src, *headers]):
            return src, ""
        cmd = [nvcc, *cflags(extra), "-c", src, "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{p.stdout}\n{p.stderr}")
        return src, p.stdout + p.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        for src, log in ex.map(compile_one, zip(srcs, objs)):
            if (verbose or ptxas_verbose) and log:
                print(f"== {os.path.basename(src)}\n{log}")

    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        libdir = os.path.join(cuda_home(nvcc), "lib64")
        cmd = [nvcc, "-shared", ARCH, "-cudart", "shared", *objs, "-o", tmp,
               "-Xlinker", f"-rpath,{libdir}"]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":  # pragma: no cover
    import sys
    print(build(verbose=True, force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv))
