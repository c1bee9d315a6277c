"""ctypes binding of the plain C++ oracle (oracle/epq_ref.cpp) -- TEST
INFRASTRUCTURE ONLY (tests, the smoke check and the bench's CPU baseline).

The shared library is compiled in-tree with the host C++ compiler by
``build()`` (``-O3 -ffp-contract=off``, no fast-math, no machine-specific
flags), so that it gives the same bits on any host.  Nothing here touches a
GPU or the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "epq_ref.cpp")
LIB = os.path.join(HERE, "libepq_ref.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle/epq_ref.cpp into oracle/libepq_ref.so (if stale)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        raise RuntimeError("no C++ compiler for the oracle")
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [cxx, "-O3", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-pthread",
           "-o", tmp, SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        c_i64, c_p = ctypes.c_int64, ctypes.c_void_p
        L.eref_f32_to_f16.argtypes = [ctypes.c_float]
        L.eref_f32_to_f16.restype = ctypes.c_uint16
        L.eref_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.eref_f16_to_f32.restype = ctypes.c_float
        L.eref_f16_of_bits.argtypes = [ctypes.c_uint32, c_i64, c_p]
        L.eref_f16_of_bits.restype = None
        L.eref_quantize.argtypes = [ctypes.c_int, c_p, c_i64, c_i64, c_p, ctypes.c_int]
        L.eref_dequantize.argtypes = [ctypes.c_int, c_p, c_i64, c_i64, c_p]
        L.eref_gemv_f64.argtypes = [ctypes.c_int, c_p, c_p, c_i64, c_i64, ctypes.c_int, c_p, c_p, ctypes.c_int]
        L.eref_gemv_f32.argtypes = [ctypes.c_int, c_p, c_p, c_i64, c_i64, ctypes.c_int, c_p, ctypes.c_int]
        L.eref_hardware_threads.argtypes = []
        for f in ("eref_quantize", "eref_dequantize", "eref_gemv_f64", "eref_gemv_f32", "eref_hardware_threads",
                  "eref_block_weights", "eref_block_bytes"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def hardware_threads() -> int:
    return int(lib().eref_hardware_threads())


def row_bytes(fmt: int, cols: int) -> int:
    bw, bb = lib().eref_block_weights(fmt), lib().eref_block_bytes(fmt)
    if bw <= 0 or cols <= 0 or cols % bw:
        return -1
    return cols // bw * bb


def quantize(fmt: int, W: np.ndarray, threads: int = 1) -> np.ndarray:
    """W float32 [rows, cols] -> packed uint8 [rows, row_bytes]."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    if W.ndim == 1:
        W = W[None, :]
    rows, cols = W.shape
    rb = row_bytes(fmt, cols)
    if rb < 0:
        raise ValueError(f"cols={cols} is not a whole number of blocks")
    out = np.empty((rows, rb), np.uint8)
    if lib().eref_quantize(fmt, _ptr(W), rows, cols, _ptr(out), int(threads)) != 0:
        raise ValueError("eref_quantize rejected the shape")
    return out


def dequantize(fmt: int, packed: np.ndarray, cols: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    rb = row_bytes(fmt, cols)
    rows = packed.size // rb
    out = np.empty((rows, cols), np.float32)
    if lib().eref_dequantize(fmt, _ptr(packed), rows, cols, _ptr(out)) != 0:
        raise ValueError("eref_dequantize rejected the shape")
    return out


def gemv_f64(fmt: int, packed: np.ndarray, x: np.ndarray, cols: int, threads: int = 1):
    """(y, bound) float64 [nvec, rows]: sum_j deq_ij x_j and sum_j |deq_ij x_j|."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    rows = packed.size // row_bytes(fmt, cols)
    nvec = x.shape[0]
    y = np.empty((nvec, rows), np.float64)
    A = np.empty((nvec, rows), np.float64)
    if lib().eref_gemv_f64(fmt, _ptr(packed), _ptr(x), rows, cols, nvec, _ptr(y), _ptr(A), int(threads)) != 0:
        raise ValueError("eref_gemv_f64 rejected the shape")
    return y, A


def gemv_f32(fmt: int, packed: np.ndarray, x: np.ndarray, cols: int, threads: int = 1, out=None):
    """float32 [nvec, rows] with float32 accumulation (the CPU baseline)."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    rows = packed.size // row_bytes(fmt, cols)
    nvec = x.shape[0]
    y = out if out is not None else np.empty((nvec, rows), np.float32)
    if lib().eref_gemv_f32(fmt, _ptr(packed), _ptr(x), rows, cols, nvec, _ptr(y), int(threads)) != 0:
        raise ValueError("eref_gemv_f32 rejected the shape")
    return y


def f16_of_bits(first: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint16)
    lib().eref_f16_of_bits(first, n, _ptr(out))
    return out
