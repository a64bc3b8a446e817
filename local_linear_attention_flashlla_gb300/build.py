"""Compile liblla.so (the C-ABI library) for sm_103a with nvcc, in tree.

Each CUDA translation unit under csrc/ is compiled in parallel to an object in
_build/, then linked into liblla.so next to this file.  No CMake, no torch
extension machinery: the library has a plain C ABI (include/lla.h).
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblla.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
           "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]


def nvcc_path():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblla.so")


def sources(sub=""):
    d = os.path.join(CSRC, sub)
    return sorted(os.path.join(d, f) for f in os.listdir(d) if f.endswith(".cu"))


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed (%d): %s\n%s" % (r.returncode, " ".join(cmd), r.stdout))
    return r.stdout


def build(verbose=False, extra_flags=()):
    """Build liblla.so; returns its path."""
    nvcc = nvcc_path()
    os.makedirs(BUILD, exist_ok=True)
    groups = {LIB: sources()}
    jobs = []
    for lib, srcs in groups.items():
        for s in srcs:
            jobs.append((lib, s, os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")))
    cmds = [[nvcc, *ARCH, *NVFLAGS, *extra_flags, "-c", s, "-o", o] for _, s, o in jobs]
    with ThreadPoolExecutor(max_workers=max(1, min(len(cmds), os.cpu_count() or 1))) as ex:
        outs = list(ex.map(_run, cmds))
    if verbose:
        for c, o in zip(cmds, outs):
            print(" ".join(c))
            if o.strip():
                print(o)
    for lib in groups:
        objs = [o for l, _, o in jobs if l == lib]
        tmp = lib + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"])
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
