"""Builds libkshipra.so in-tree with nvcc for sm_103a.

The translation units compile in parallel (one nvcc per file) and are linked
into ``paged_kv_cache_arena_gb300/libkshipra.so`` with the static CUDA
runtime.  Objects go to ``_build/`` at the repository root.
"""

from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libkshipra.so")
SOURCES = ("api.cu", "append_rope.cu", "decode.cu", "prefill.cu", "prefill_pair.cu", "noalloc.cu", "blocks.cu",
           "prefix_cache.cpp")
HEADERS = ("common.cuh", "internal.h", "rope.cuh")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "kshipra.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    procs = []
    for src in SOURCES:
        obj = os.path.join(OBJ, os.path.splitext(src)[0] + ".o")
        cmd = [NVCC, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    objs, errors = [], []
    for src, obj, p in procs:
        out, _ = p.communicate()
        if p.returncode:
            errors.append("%s:\n%s" % (src, out.decode(errors="replace")))
        objs.append(obj)
    if errors:
        raise RuntimeError("nvcc failed\n" + "\n".join(errors))
    tmp = LIB + ".%d.tmp" % os.getpid()
    subprocess.check_call([NVCC, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
