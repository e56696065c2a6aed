"""Seeded, counter-based synthetic input generator (host and device).

This package produces every synthetic input of the decode-step workloads:
weights, pre-filled KV-cache contents, prompt/start tokens and per-slot start
positions.  It holds none of the decode step's arithmetic.  Host values come
from ``libsynth_host.so`` and device fills from ``libsynth_cuda.so``; both are
compiled from the same header (``synth.h``), so a value depends only on
(seed, tensor kind, layer, sub-index, element index) and is bitwise equal on
CPU and GPU.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_DIR, "libsynth_host.so")
CUDA_LIB = os.path.join(_DIR, "libsynth_cuda.so")

F32, BF16, Q8, Q4 = 0, 1, 2, 3

TOK_EMBD, ATTN_NORM, WQ, WK, WV, WO, FFN_NORM = 1, 2, 3, 4, 5, 6, 7
WGATE, WUP, WDOWN, WROUTER, OUT_NORM, OUTPUT = 8, 9, 10, 11, 12, 13
KCACHE, VCACHE, TOKENS, POSITIONS = 14, 15, 16, 17
BQ, BK, BV = 18, 19, 20   # q / k / v bias vectors


def build_commands(cuda_arch: str = "103a"):
    """Compiler command lines that build this package's shared libraries."""
    host = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-o", HOST_LIB,
            os.path.join(_DIR, "synth_host.c"), "-lm"]
    dev = ["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC", "-std=c++17", "-fmad=false",
           f"-gencode=arch=compute_{cuda_arch},code=sm_{cuda_arch}",
           "-o", CUDA_LIB, os.path.join(_DIR, "synth_cuda.cu")]
    return [host, dev]


_host_lib = None
_cuda_lib = None


def _host():
    global _host_lib
    if _host_lib is None:
        if not os.path.exists(HOST_LIB):
            raise RuntimeError(f"{HOST_LIB} is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(HOST_LIB)
        u64, i64, u32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_uint32
        p = ctypes.c_void_p
        lib.synth_host_key.restype = u64
        lib.synth_host_key.argtypes = [u64, u32, u32, u32]
        lib.synth_host_fill_f32.argtypes = [p, u64, u64, i64, ctypes.c_float, ctypes.c_int]
        lib.synth_host_fill_bf16.argtypes = [p, u64, u64, i64, ctypes.c_float]
        lib.synth_host_fill_ih12.argtypes = [p, u64, u64, i64]
        lib.synth_host_fill_uniform_int.argtypes = [p, u64, u64, i64, i64, u32]
        lib.synth_host_words.argtypes = [p, u64, u64, i64]
        lib.synth_host_f32_to_bf16.restype = ctypes.c_uint16
        lib.synth_host_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.synth_host_fill_q8_rows.argtypes = [p, p, u64, i64, i64, i64, ctypes.c_float]
        lib.synth_host_fill_q4_rows.argtypes = [p, p, u64, i64, i64, i64, ctypes.c_float]
        lib.synth_host_f32_to_f16.restype = ctypes.c_uint16
        lib.synth_host_f32_to_f16.argtypes = [ctypes.c_float]
        lib.synth_host_f16_to_f32.restype = ctypes.c_float
        lib.synth_host_f16_to_f32.argtypes = [ctypes.c_uint16]
        _host_lib = lib
    return _host_lib


def _cuda():
    global _cuda_lib
    if _cuda_lib is None:
        if not os.path.exists(CUDA_LIB):
            raise RuntimeError(f"{CUDA_LIB} is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(CUDA_LIB)
        u64, i64, u32, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_uint32, ctypes.c_int
        p, f = ctypes.c_void_p, ctypes.c_float
        lib.synth_dev_fill_matrix.argtypes = [p, i32, i64, i64, i64, i64, u64, f, p]
        lib.synth_dev_fill_const.argtypes = [p, i32, i64, f, p]
        lib.synth_dev_fill_kv.argtypes = [p, i32, i32, i64, i32, i64, i64, u64, f, p]
        lib.synth_dev_fill_uniform_int.argtypes = [p, i64, u64, u64, i64, u32, p]
        for fn in (lib.synth_dev_fill_matrix, lib.synth_dev_fill_const, lib.synth_dev_fill_kv,
                   lib.synth_dev_fill_uniform_int):
            fn.restype = i32
        _cuda_lib = lib
    return _cuda_lib


# ------------------------------------------------------------------ host side

def key(seed: int, kind: int, layer: int = 0, sub: int = 0) -> int:
    """Stream key of one logical tensor."""
    return int(_host().synth_host_key(seed, kind, layer, sub))


def values(k: int, idx0: int, n: int, sigma: float, dtype: int) -> np.ndarray:
    """Generated elements idx0 .. idx0+n-1, rounded to ``dtype``, as float32."""
    out = np.empty(n, dtype=np.float32)
    _host().synth_host_fill_f32(out.ctypes.data, k, idx0, n, sigma, dtype)
    return out


def bf16_bits(k: int, idx0: int, n: int, sigma: float) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    _host().synth_host_fill_bf16(out.ctypes.data, k, idx0, n, sigma)
    return out


def ih12(k: int, idx0: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _host().synth_host_fill_ih12(out.ctypes.data, k, idx0, n)
    return out


def uniform_int(k: int, idx0: int, n: int, lo: int, count: int) -> np.ndarray:
    """Integers uniform in [lo, lo + count)."""
    out = np.empty(n, dtype=np.int64)
    _host().synth_host_fill_uniform_int(out.ctypes.data, k, idx0, n, lo, count)
    return out


def words(k: int, n0: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _host().synth_host_words(out.ctypes.data, k, n0, n)
    return out


def f32_to_bf16_bits(x: float) -> int:
    return int(_host().synth_host_f32_to_bf16(x))


def f32_to_f16_bits(x: float) -> int:
    return int(_host().synth_host_f32_to_f16(x))


def f16_to_f32(h: int) -> float:
    return float(_host().synth_host_f16_to_f32(h))


def q8_rows(k: int, row0: int, nrows: int, cols: int, sigma: float):
    """Q8 rows [row0, row0 + nrows) of a [.][cols] matrix: (the row bytes in the
    library's layout, uint8 [nrows][cols + cols / 16]; the weights d * q, fp32)."""
    raw = np.empty((nrows, cols + cols // 16), dtype=np.uint8)
    w = np.empty((nrows, cols), dtype=np.float32)
    _host().synth_host_fill_q8_rows(raw.ctypes.data, w.ctypes.data, k, row0, nrows, cols, sigma)
    return raw, w


def q4_rows(k: int, row0: int, nrows: int, cols: int, sigma: float):
    """Q4 rows [row0, row0 + nrows) of a [.][cols] matrix: (the row bytes in the
    library's layout, uint8 [nrows][cols / 2 + cols / 16]; the weights d * (u - 8),
    fp32)."""
    raw = np.empty((nrows, cols // 2 + cols // 16), dtype=np.uint8)
    w = np.empty((nrows, cols), dtype=np.float32)
    _host().synth_host_fill_q4_rows(raw.ctypes.data, w.ctypes.data, k, row0, nrows, cols, sigma)
    return raw, w


# ---------------------------------------------------------------- device side

def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"{what} failed with CUDA error {rc}")


def dev_fill_matrix(ptr: int, dtype: int, row0: int, row_step: int, rows: int, cols: int,
                    k: int, sigma: float, stream: int = 0):
    """Logical row r of a [rows][cols] tensor -> device row row0 + r*row_step."""
    _check(_cuda().synth_dev_fill_matrix(ptr, dtype, row0, row_step, rows, cols, k, sigma, stream),
           "synth_dev_fill_matrix")


def dev_fill_const(ptr: int, dtype: int, n: int, value: float, stream: int = 0):
    _check(_cuda().synth_dev_fill_const(ptr, dtype, n, value, stream), "synth_dev_fill_const")


def dev_fill_kv(ptr: int, dtype: int, n_kv: int, cap: int, hd: int, j_lo: int, j_hi: int,
                k: int, sigma: float, stream: int = 0):
    """Positions [j_lo, j_hi) of a [n_kv][cap][hd] cache block (slot = j % cap)."""
    _check(_cuda().synth_dev_fill_kv(ptr, dtype, n_kv, cap, hd, j_lo, j_hi, k, sigma, stream),
           "synth_dev_fill_kv")


def dev_fill_uniform_int(ptr: int, n: int, k: int, idx0: int, lo: int, count: int,
                         stream: int = 0):
    _check(_cuda().synth_dev_fill_uniform_int(ptr, n, k, idx0, lo, count, stream),
           "synth_dev_fill_uniform_int")
