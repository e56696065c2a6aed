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


def build_jobs():
    """(output, inputs, command) triples; empty until the CUDA sources exist."""
    srcs = sources()
    if not srcs:
        return []
    cmd = ["nvcc", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-lineinfo",
           f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}", "-I", os.path.join(ROOT, "include"),
           "-I", CSRC, "-o", LIB] + srcs
    return [(LIB, srcs + headers(), cmd)]
