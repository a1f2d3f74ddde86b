"""Build the C-ABI library ``libzero_step.so`` in-tree for sm_103a.

nvcc compiles the CUDA translation units for ``compute_103a``/``sm_103a`` only
(no PTX for other targets, so the library runs on GB300-class parts only),
g++ compiles the host-only layout code, and nvcc links both into one shared
library with the CUDA runtime linked statically.  Translation units compile
in parallel; nothing is rebuilt when the library is newer than every source.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libzero_step.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "-Xptxas", "-v", "--expt-relaxed-constexpr"]
# host C++: IEEE binary32 with no multiply-add contraction (GCC contracts by
# default on AArch64), sqrt without errno so the host Adam loops vectorise
CXX_FLAGS = ["-O3", "-std=c++17", "-fPIC", "-Wall", "-Wextra", "-ffp-contract=off",
             "-fno-math-errno", "-pthread"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libzero_step.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cpp", ".cuh", ".h")))


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)] + [__file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link ``libzero_step.so``; returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    objs = []
    for src in sources():
        name, ext = os.path.splitext(os.path.basename(src))
        if ext not in (".cu", ".cpp"):
            continue
        obj = os.path.join(BUILD, name + ".o")
        objs.append(obj)
        if ext == ".cu":
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-c", src, "-o", obj]
        else:
            cmd = ["g++", *CXX_FLAGS, "-I", INCLUDE, "-c", src, "-o", obj]
        log = open(obj + ".log", "w")
        jobs.append((cmd, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log, obj))
    failed = []
    for cmd, proc, log, obj in jobs:
        rc = proc.wait()
        log.close()
        if rc != 0 or verbose:
            with open(obj + ".log") as f:
                sys.stderr.write(f.read())
        if rc != 0:
            failed.append(" ".join(cmd))
    if failed:
        raise RuntimeError("compilation failed:\n" + "\n".join(failed))
    tmp = LIB + ".tmp"
    subprocess.run([nvcc, *ARCH, "-shared", "-Xcompiler", "-pthread", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
