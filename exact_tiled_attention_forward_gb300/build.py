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
# FA_DEBUG build of libfa (device-side bounds checks that report instead of
# touching memory out of range): a separate library, never the one the
# binding loads by default
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libfa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa")


def sources(folder=CSRC):
    return sorted(os.path.join(folder, f) for f in os.listdir(folder) if f.endswith(".cu"))


def _stale(outputs=(LIB, LIB_SINGLE_GPU)) -> bool:
    if not all(os.path.exists(o) for o in outputs):
        return True
    t = min(os.path.getmtime(o) for o in outputs)
    deps = sources() + sources(CSRC_SINGLE)
    for folder in (CSRC, CSRC_SINGLE, INCLUDE):
        deps += [os.path.join(folder, f) for f in os.listdir(folder) if f.endswith((".cuh", ".h"))]
    return any(os.path.getmtime(f) > t for f in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile and link both libraries if any source is newer than them; return
    libfa.so's path. debug=True builds only the FA_DEBUG libfa (_build_debug/)."""
    out_dir = BUILD_DEBUG if debug else BUILD
    outputs = (LIB_DEBUG,) if debug else (LIB, LIB_SINGLE_GPU)
    if not force and not _stale(outputs):
        return outputs[0]
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    flags = [*FLAGS, *extra_flags] + (["-DFA_DEBUG"] if debug else [])

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    base, single = sources(), ([] if debug else sources(CSRC_SINGLE))
    with concurrent.futures.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        objs = list(ex.map(compile_one, base + single))
    base_objs, single_objs = objs[:len(base)], objs[len(base):]
    links = ((LIB_DEBUG, base_objs),) if debug else ((LIB, base_objs), (LIB_SINGLE_GPU, base_objs + single_objs))
    for out, parts in links:
        tmp = out + ".tmp"
        cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *parts]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {os.path.basename(out)} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)
    return outputs[0]


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
