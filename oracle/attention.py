"""Decode-step attention oracle (test infrastructure only).

"smolmaxxing", compute table, row "带阈值的 Q8_0 注意力": the key/value cache
holds Q8_0 blocks; all key dot products of a step are computed first, so the
softmax maximum M is known; positions whose score is below M + ln(1e-4) are
skipped (no exponential, no value row); the rest are weighted by
exp(s - M) / sum exp(s - M) over the kept positions.

Readings where the page is silent (listed in the design notes):

* scores are s_p = scale * q . k_p with the keys as the Q8_0 cache holds
  them (dequantized), scale = 1/sqrt(head_dim) in the decode steps;
* the threshold is inclusive (s_p >= M + skip_log is kept), skip_log =
  ln(1e-4) by default and -inf keeps every position;
* grouped heads: query head hq uses key/value head hq // group;
* the step's own key and value are quantized to Q8_0 (the format oracle's
  quantizer) and appended at position `pos` before the step attends over
  positions 0..pos.

float64 throughout, except that the skip decision and the weights may be
taken on given float32 scores (the GPU's), so that the rule is applied to the
same numbers on both sides.
"""
from __future__ import annotations

import math

import numpy as np

from .formats import Q8_0, dequantize, quantize

SKIP_LOG = math.log(1e-4)


def q8_rows(x: np.ndarray) -> np.ndarray:
    """Q8_0 values of rows x [n, D] (quantize then dequantize, float32)."""
    x = np.asarray(x, np.float32)
    return dequantize(Q8_0, quantize(Q8_0, x), x.shape[1])


def attention_f64(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, skip_log: float = SKIP_LOG,
                  scores: np.ndarray | None = None):
    """One key/value head: q [G, D], K, V [T, D] (cache values).

    Returns (out [G, D], scores [G, T], kept [G, T] bool)."""
    q = np.asarray(q, np.float64)
    if scores is None:
        s = float(scale) * (q @ np.asarray(K, np.float64).T)
    else:
        s = np.asarray(scores, np.float64)
    M = s.max(axis=1, keepdims=True)
    kept = s >= M + skip_log
    w = np.where(kept, np.exp(s - M), 0.0)
    out = (w @ np.asarray(V, np.float64)) / w.sum(axis=1, keepdims=True)
    return out, s, kept


def decode_attention_f64(q: np.ndarray, K: np.ndarray, V: np.ndarray, n_heads: int, scale: float,
                         skip_log: float = SKIP_LOG, scores: np.ndarray | None = None):
    """All heads: q [n_heads, D]; K, V [n_kv, T, D] -> out [n_heads, D]."""
    n_kv = K.shape[0]
    G = n_heads // n_kv
    out = np.empty((n_heads, q.shape[1]))
    for h in range(n_kv):
        sc = None if scores is None else scores[h * G:(h + 1) * G]
        out[h * G:(h + 1) * G] = attention_f64(q[h * G:(h + 1) * G], K[h], V[h], scale, skip_log, sc)[0]
    return out
