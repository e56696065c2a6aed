"""Compiler jobs for the decode-step library (no imports of the library itself)."""
from __future__ import annotations

import glob
import os

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libpnb.so")
ARCH = "103a"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h")))


OBJ = os.path.join(PKG, "_objs")
FLAGS = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-lineinfo",
         f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}"]


def build_jobs():
    """Build stages: a list of parallel (output, inputs, command) jobs per stage -
    one object per CUDA source, then the shared-library link."""
    srcs = sources()
    if not srcs:
        return []
    objs, compile_jobs = [], []
    for src in srcs:
        obj = os.path.join(OBJ, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        compile_jobs.append((obj, [src] + headers(),
                             ["nvcc"] + FLAGS + ["-I", os.path.join(ROOT, "include"), "-I", CSRC,
                                                 "-c", src, "-o", obj]))
    link = (LIB, objs, ["nvcc", "-shared", f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}",
                        "-o", LIB] + objs)
    return [compile_jobs, [link]]
