"""Builds libzero_pml.so in-tree with nvcc for sm_103a (GB300).

The translation units are compiled in parallel -- the host-only parts
(layout, error strings, state init; the offload step on the host cores) with
g++ and the CUDA part (kernels and device entry points) with nvcc -- and
linked against the shared CUDA runtime, so that the library and PyTorch share
one runtime (one current device, one set of streams).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libzero_pml.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "bin", "nvcc")):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libzero_pml.so")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cpp", ".h", ".cuh")))


def _up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    deps = _sources() + [os.path.join(INCLUDE, "zero_pml.h"), os.path.abspath(__file__)]
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles the library if a source is newer than it; returns its path."""
    if not force and _up_to_date():
        return LIB
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    os.makedirs(BUILD, exist_ok=True)
    common = ["-std=c++17", "-O3", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    cu_flags = ARCH + ["-lineinfo", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
                       "--expt-relaxed-constexpr", "-Xptxas", "-v" if verbose else "-O3"]
    jobs = []
    objs = []
    for src in _sources():
        if src.endswith((".h", ".cuh")):
            continue
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        objs.append(obj)
        if src.endswith(".cu"):
            jobs.append([nvcc, "-c", src, "-o", obj] + common + cu_flags)
        else:
            # host code: binary32 evaluated as written (no FMA contraction);
            # no errno from sqrt, so that its loops vectorise (results unchanged)
            jobs.append(["g++", "-c", src, "-o", obj, "-std=c++17", "-O3", "-fPIC", "-pthread",
                         "-ffp-contract=off", "-fno-fast-math", "-fno-math-errno", "-Wall",
                         "-I", INCLUDE, "-I", CSRC])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {cmd[2]}")
    tmp = LIB + f".tmp{os.getpid()}"
    link = [nvcc, "-shared", "-cudart", "shared"] + ARCH + ["-o", tmp] + objs + [
        "-Xcompiler", "-pthread",
        "-Xlinker", "-rpath," + os.path.join(cuda, "lib64"), "-Xlinker", "-rpath,$ORIGIN"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(" ".join(link) + "\n" + r.stdout + r.stderr)
        raise RuntimeError("link of libzero_pml.so failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
