"""Dequant-GEMV oracle (test infrastructure only).

Handbook page "端侧推理：llama.cpp 与 GGUF、MLX、ExecuTorch", section
"速度上限：带宽 ÷ 权重字节数": a batch-1 decode step multiplies every weight
matrix by one activation vector; with several speculative tokens the same
weights multiply several vectors.  The reference value is the plain
definition ``y[v, i] = sum_j deq(W)[i, j] * x[v, j]`` in float64, with the
companion magnitude ``A[v, i] = sum_j |deq(W)[i, j] * x[v, j]|`` that scales
the accepted error.
"""
from __future__ import annotations

import numpy as np

from .formats import dequantize


def _as2d(x):
    x = np.asarray(x)
    return x[None, :] if x.ndim == 1 else x


def gemv_f64(fmt: int, packed: np.ndarray, x: np.ndarray, cols: int) -> np.ndarray:
    """x [nvec, cols] -> y [nvec, rows] float64."""
    W = dequantize(fmt, packed, cols).astype(np.float64)
    return _as2d(x).astype(np.float64) @ W.T


def gemv_bound(fmt: int, packed: np.ndarray, x: np.ndarray, cols: int) -> np.ndarray:
    """A [nvec, rows] = sum_j |deq(W)_ij * x_j| in float64."""
    W = np.abs(dequantize(fmt, packed, cols).astype(np.float64))
    return np.abs(_as2d(x).astype(np.float64)) @ W.T
