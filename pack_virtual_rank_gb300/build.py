"""Build ``librelay.so`` in-tree with nvcc for sm_103a (GB300).

Every translation unit compiles in parallel into ``_build/``; the shared library is
linked next to this file. No cmake, no torch extension machinery: the library is a
plain C ABI (``include/relay.h``).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "librelay.so")

SOURCES = ["plan.cpp", "program.cpp", "chain.cpp", "abi.cpp", "passes.cu", "chain_kernel.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the relay library needs the CUDA toolkit to build")


def _flags(verbose_ptxas: bool = False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-Xcompiler", "-fPIC",
                "-Xcompiler", "-Wall", "-I", INCLUDE, "-I", CSRC]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + [os.path.join(CSRC, "program.h"),
                                                       os.path.join(CSRC, "device.cuh"),
                                                       os.path.join(INCLUDE, "relay.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile and link the library if any source is newer than it; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    jobs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        jobs.append(([cc, "-c", os.path.join(CSRC, src), "-o", obj] + _flags(verbose_ptxas), obj))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        logs = list(ex.map(run, [j[0] for j in jobs]))
    if verbose_ptxas:
        sys.stderr.write("".join(logs))
    tmp = LIB + f".tmp{os.getpid()}"
    run([cc, "-shared"] + ARCH + ["-o", tmp] + [j[1] for j in jobs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
