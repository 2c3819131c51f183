"""Build the k3huf shared library in-tree for sm_103a.

Compiles ``csrc/*.cu`` with nvcc (``-gencode arch=compute_103a,code=sm_103a``)
and ``csrc/*.cpp`` with g++, in parallel, and links
``_build/libk3huf.so`` against the shared CUDA runtime.  No cmake, no torch
extension machinery: the library has a plain C ABI (``include/k3huf.h``).
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libk3huf.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _cuda_home() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _sources():
    cu = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cpp"))
    hdr = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".h"))
    return cu, cpp, hdr + [os.path.join(INCLUDE, "k3huf.h")]


def _stale(target, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_nvcc=()) -> str:
    """Compile (when stale) and return the library path."""
    cu, cpp, hdrs = _sources()
    os.makedirs(BUILD, exist_ok=True)
    if not force and not _stale(LIB, cu + cpp + hdrs + [os.path.abspath(__file__)]):
        return LIB
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    inc = ["-I", INCLUDE, "-I", CSRC]
    jobs = []
    for src in cu:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        jobs.append([nvcc, ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "--expt-relaxed-constexpr", *inc, *extra_nvcc, "-c", src, "-o", obj])
    for src in cpp:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        jobs.append(["g++", "-O2", "-std=c++17", "-fPIC", "-pthread", "-Wall", *inc, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return cmd[-1]

    with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(run, jobs))
    tmp = LIB + f".{os.getpid()}.tmp"
    libdir = os.path.join(cuda, "lib64")
    if not os.path.isdir(libdir):
        libdir = os.path.join(cuda, "lib")
    link = [nvcc, ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs, "-lpthread",
            "-Xlinker", f"-rpath={libdir}"]
    run(link)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
