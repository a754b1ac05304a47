"""Build the in-tree C-ABI library libzero_step.so for sm_103a.

Two translation units (the CUDA kernels + entry points, and the host-only
plan code) are compiled in parallel by nvcc and linked into one shared
library with the CUDA runtime linked statically, so the library needs no
libcudart at load time and can be loaded (and its host-only entry points
called) on a machine without a GPU.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libzero_step.so")
BUILD_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]
SOURCES = [os.path.join(CSRC, "zero_step.cu"), os.path.join(CSRC, "plan.cpp"),
           os.path.join(CSRC, "ckpt.cpp")]
HEADERS = [os.path.join(INCLUDE, "zero_step.h")] + sorted(
    os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh"))


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in SOURCES + HEADERS + [__file__])


def compile_commands():
    os.makedirs(BUILD_DIR, exist_ok=True)
    cmds, objs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        cmds.append([nvcc(), *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj])
        objs.append(obj)
    link = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", LIB + ".tmp", *objs]
    return cmds, link


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    cmds, link = compile_commands()
    procs = [subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
             for c in cmds]
    failed = []
    for c, p in zip(cmds, procs):
        out, _ = p.communicate()
        if verbose and out:
            sys.stdout.write(out)
        if p.returncode != 0:
            failed.append((c, out))
    if failed:
        msg = "\n".join(f"$ {' '.join(c)}\n{o}" for c, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    subprocess.run(link, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
