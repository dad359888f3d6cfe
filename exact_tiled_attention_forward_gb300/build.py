"""Build ``libfa.so`` (the CUDA library behind the C ABI in ``include/fa.h``)
and ``libfa_single_gpu.so`` (the same objects plus the cluster-multicast
forward of ``include/fa_single_gpu.h``, for processes that use one GPU).

Each ``.cu`` file is compiled for sm_103a in its own ``nvcc`` process (in
parallel), then linked into shared libraries with the CUDA runtime linked
statically, so they depend on nothing but the driver. ``libfa.so`` is linked
from ``csrc/`` alone, so it holds no multicast code. The results go to
``_build/`` inside this package directory.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
CSRC_SINGLE = os.path.join(PKG, "csrc_single_gpu")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libfa.so")
LIB_SINGLE_GPU = os.path.join(BUILD, "libfa_single_gpu.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa")


def sources(folder=CSRC):
    return sorted(os.path.join(folder, f) for f in os.listdir(folder) if f.endswith(".cu"))


def _stale() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(LIB_SINGLE_GPU)):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(LIB_SINGLE_GPU))
    deps = sources() + sources(CSRC_SINGLE)
    for folder in (CSRC, CSRC_SINGLE, INCLUDE):
        deps += [os.path.join(folder, f) for f in os.listdir(folder) if f.endswith((".cuh", ".h"))]
    return any(os.path.getmtime(f) > t for f in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link both libraries if any source is newer than them; return libfa.so's path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    base, single = sources(), sources(CSRC_SINGLE)
    with concurrent.futures.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        objs = list(ex.map(compile_one, base + single))
    base_objs, single_objs = objs[:len(base)], objs[len(base):]
    for out, parts in ((LIB, base_objs), (LIB_SINGLE_GPU, base_objs + single_objs)):
        tmp = out + ".tmp"
        cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *parts]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {os.path.basename(out)} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
