"""Build libgcsgd.so in-tree with nvcc for sm_103a (GB300).

Each .cu file compiles in parallel to an object under ``_build/``; the
objects link into ``gradient_compression_sgd_gb300/libgcsgd.so`` against the
shared CUDA runtime.  Rebuilds only when a source or header is newer than the
library.  Usage: ``python -m gradient_compression_sgd_gb300.build [--force]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libgcsgd.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "--extended-lambda", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-O2", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin on PATH)")


def cuda_lib_dir(nv: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nv))), "lib64")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    nv = nvcc()
    os.makedirs(BUILD, exist_ok=True)
    jobs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        jobs.append((src, obj, [nv, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]))
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        futs = {ex.submit(subprocess.run, cmd, capture_output=True, text=True): src for src, _, cmd in jobs}
        for f in cf.as_completed(futs):
            r = f.result()
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {futs[f]}:\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout, r.stderr, file=sys.stderr)
    libdir = cuda_lib_dir(nv)
    tmp = LIB + f".{os.getpid()}.tmp"
    link = [nv, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *[o for _, o, _ in jobs],
            "-Xlinker", f"-rpath,{libdir}", "-L", libdir]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
