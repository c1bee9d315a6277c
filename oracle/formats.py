"""Block formats: quantizers, canonical byte layouts and dequantizers.

Oracle code (test infrastructure only).  Follows the handbook page
"端侧推理：llama.cpp 与 GGUF、MLX、ExecuTorch", section "GGUF 的量化格式":

* Q8_0: blocks of 32 weights, one fp16 scale, symmetric int8 codes;
  the scale maps the largest magnitude to 127.
* Q4_0: blocks of 32, one fp16 scale chosen from the signed value of largest
  magnitude so that this value lands on code -8; codes -8..7 stored with a
  +8 offset.
* Q4_1: blocks of 32, fp16 scale and fp16 minimum, codes 0..15.
* Q4_K (the page's simplified variant): superblocks of 256 made of 8
  sub-blocks of 32.  Each sub-block has its own scale (range/15) and min
  (minus the sub-block minimum, the minimum first clamped to <= 0); both are
  coded in 6 bits against two fp16 superblock factors (largest scale / 63
  and largest min / 63).  Scale codes are kept in 1..63, min codes in 0..63.

Readings where the page is silent (each is listed in the design notes):

1. All quantizer arithmetic is IEEE float32: true division, ``rint`` with
   ties to even, clamp in float before the integer cast.
2. Codes are computed against the *stored* fp16 factors (the page counts
   16 bits for each factor but divides by the unrounded float32 value).
3. A zero factor gives all-zero codes (the page's listing would divide by
   zero and produce NaN); for Q4_K a zero ``d`` gives scale codes of 1 and
   a zero ``dmin`` gives min codes of 0.
4. Q4_0's "largest magnitude" takes the first index on ties.
5. Byte layout (the page fixes sizes only; this is the project's own
   definition, not a claim of file compatibility):
     Q8_0  34 B = f16 d | int8 q[32]
     Q4_0  18 B = f16 d | u8 qs[16]
     Q4_1  20 B = f16 d | f16 m | u8 qs[16]
     Q4_K 144 B = f16 d | f16 dmin | u8 scales[12] | u8 qs[128]
   fp16 values little-endian; weight j of a 32-run sits in byte j>>1, low
   nibble when j is even; Q4_K sub-block s owns qs[16s:16s+16]; the 16
   six-bit codes (8 scale codes then 8 min codes) form a little-endian
   96-bit stream, code t at bits 6t..6t+5.  Rows are contiguous and blocks
   run in column order within a row.
6. Signed zeros: inputs are first mapped ``x -> x + 0`` (so -0 becomes +0)
   and the Q4_K min is formed as ``0 - lo``; every max/min then has one
   well-defined result and a zero factor is always +0 (Q4_0's factor of an
   all-zero block is +0 / -8 = -0, kept as the division gives it).
   Inputs must be finite.
"""
from __future__ import annotations

import numpy as np

Q8_0, Q4_0, Q4_1, Q4_K = 0, 1, 2, 3
FORMATS = (Q8_0, Q4_0, Q4_1, Q4_K)
NAMES = {Q8_0: "Q8_0", Q4_0: "Q4_0", Q4_1: "Q4_1", Q4_K: "Q4_K"}
BLOCK_WEIGHTS = {Q8_0: 32, Q4_0: 32, Q4_1: 32, Q4_K: 256}
BLOCK_BYTES = {Q8_0: 34, Q4_0: 18, Q4_1: 20, Q4_K: 144}

_F32 = np.float32


def row_bytes(fmt: int, cols: int) -> int:
    """Packed bytes of one row, or -1 when cols is not a whole number of blocks."""
    bw = BLOCK_WEIGHTS[fmt]
    if cols <= 0 or cols % bw:
        return -1
    return cols // bw * BLOCK_BYTES[fmt]


def bits_per_weight(fmt: int) -> float:
    return 8.0 * BLOCK_BYTES[fmt] / BLOCK_WEIGHTS[fmt]


# ---------------------------------------------------------------- fp16 helpers
def _f16(v: np.ndarray) -> np.ndarray:
    """float32 -> IEEE binary16, round to nearest even (numpy's conversion)."""
    return np.asarray(v, dtype=_F32).astype(np.float16)


def _F(h: np.ndarray) -> np.ndarray:
    """Exact float32 value of an fp16."""
    return np.asarray(h, dtype=np.float16).astype(_F32)


def _f16_bytes(h: np.ndarray) -> np.ndarray:
    """[n] fp16 -> [n, 2] little-endian bytes."""
    return np.ascontiguousarray(h.astype("<f2")).view(np.uint8).reshape(-1, 2)


def _f16_from_bytes(b: np.ndarray) -> np.ndarray:
    """[n, 2] little-endian bytes -> [n] fp16."""
    return np.ascontiguousarray(b).view("<f2").reshape(-1).astype(np.float16)


def _rint_clip(num: np.ndarray, den: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """clamp(rint(num / den), lo, hi) in float32; 0 where den == 0."""
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(np.asarray(num, _F32) / np.asarray(den, _F32))
    q = np.clip(q, _F32(lo), _F32(hi))
    q = np.where(np.asarray(den) == 0, _F32(0), q)
    return q


def _pack_nibbles(n: np.ndarray) -> np.ndarray:
    """[..., 32] codes 0..15 -> [..., 16] bytes; even index in the low nibble."""
    n = n.astype(np.uint8)
    return (n[..., 0::2] | (n[..., 1::2] << 4)).astype(np.uint8)


def _unpack_nibbles(b: np.ndarray) -> np.ndarray:
    """[..., 16] bytes -> [..., 32] codes."""
    out = np.empty(b.shape[:-1] + (32,), dtype=np.uint8)
    out[..., 0::2] = b & 0x0F
    out[..., 1::2] = b >> 4
    return out


# ---------------------------------------------------------------- Q8_0
def _quant_q8_0(b: np.ndarray):
    """b: [nb, 32] float32 -> (d fp16 [nb], q int8 [nb, 32])."""
    amax = np.max(np.abs(b), axis=1)
    d = _f16(amax / _F32(127.0))
    q = _rint_clip(b, _F(d)[:, None], -127, 127)
    return d, q.astype(np.int8)


def _pack_q8_0(d, q):
    out = np.empty((d.shape[0], 34), np.uint8)
    out[:, 0:2] = _f16_bytes(d)
    out[:, 2:34] = q.view(np.uint8)
    return out


def _deq_q8_0(blk: np.ndarray) -> np.ndarray:
    d = _F(_f16_from_bytes(blk[:, 0:2]))
    q = np.ascontiguousarray(blk[:, 2:34]).view(np.int8).astype(_F32)
    return d[:, None] * q


# ---------------------------------------------------------------- Q4_0
def _quant_q4_0(b: np.ndarray):
    i_star = np.argmax(np.abs(b), axis=1)            # first index on ties
    vmax = b[np.arange(b.shape[0]), i_star]          # signed value
    d = _f16(vmax / _F32(-8.0))
    q = _rint_clip(b, _F(d)[:, None], -8, 7)
    return d, (q + _F32(8)).astype(np.uint8)


def _pack_q4_0(d, n):
    out = np.empty((d.shape[0], 18), np.uint8)
    out[:, 0:2] = _f16_bytes(d)
    out[:, 2:18] = _pack_nibbles(n)
    return out


def _deq_q4_0(blk):
    d = _F(_f16_from_bytes(blk[:, 0:2]))
    n = _unpack_nibbles(blk[:, 2:18]).astype(_F32)
    return d[:, None] * (n - _F32(8))


# ---------------------------------------------------------------- Q4_1
def _quant_q4_1(b: np.ndarray):
    lo = np.min(b, axis=1)
    hi = np.max(b, axis=1)
    d = _f16((hi - lo) / _F32(15.0))
    m = _f16(lo)
    n = _rint_clip(b - _F(m)[:, None], _F(d)[:, None], 0, 15)
    return d, m, n.astype(np.uint8)


def _pack_q4_1(d, m, n):
    out = np.empty((d.shape[0], 20), np.uint8)
    out[:, 0:2] = _f16_bytes(d)
    out[:, 2:4] = _f16_bytes(m)
    out[:, 4:20] = _pack_nibbles(n)
    return out


def _deq_q4_1(blk):
    d = _F(_f16_from_bytes(blk[:, 0:2]))
    m = _F(_f16_from_bytes(blk[:, 2:4]))
    n = _unpack_nibbles(blk[:, 4:20]).astype(_F32)
    return n * d[:, None] + m[:, None]


# ---------------------------------------------------------------- Q4_K
def _quant_q4_k(b: np.ndarray):
    """b: [nsb, 8, 32] float32 superblocks.

    Returns (d, dmin) fp16 [nsb], (c, k) uint8 [nsb, 8], n uint8 [nsb, 8, 32].
    """
    lo = np.minimum(np.min(b, axis=2), _F32(0))      # sub-block minimum, clamped <= 0
    hi = np.max(b, axis=2)
    sc = (hi - lo) / _F32(15.0)                       # sub-block scale
    mn = _F32(0) - lo                                 # sub-block min (+0 when lo is 0)
    d = _f16(np.max(sc, axis=1) / _F32(63.0))
    dmin = _f16(np.max(mn, axis=1) / _F32(63.0))
    dF, dminF = _F(d)[:, None], _F(dmin)[:, None]
    c = _rint_clip(sc, dF, 1, 63)
    c = np.where(dF == 0, _F32(1), c)                 # reading 3: zero d -> code 1
    k = _rint_clip(mn, dminF, 0, 63)
    S = dF * c                                        # exact: 11 x 6 significant bits
    M = dminF * k
    n = _rint_clip(b + M[:, :, None], S[:, :, None], 0, 15)
    return d, dmin, c.astype(np.uint8), k.astype(np.uint8), n.astype(np.uint8)


def _pack_scales(c: np.ndarray, k: np.ndarray) -> np.ndarray:
    """16 six-bit codes (c_0..c_7, k_0..k_7) -> 12 bytes, little-endian stream."""
    codes = np.concatenate([c, k], axis=1).astype(np.uint64)   # [n, 16]
    out = np.zeros((codes.shape[0], 12), np.uint8)
    for t in range(16):
        for bit in range(6):
            pos = 6 * t + bit
            v = ((codes[:, t] >> np.uint64(bit)) & np.uint64(1)).astype(np.uint8)
            out[:, pos // 8] |= (v << (pos % 8)).astype(np.uint8)
    return out


def _unpack_scales(s: np.ndarray):
    codes = np.zeros((s.shape[0], 16), np.uint8)
    for t in range(16):
        for bit in range(6):
            pos = 6 * t + bit
            v = (s[:, pos // 8] >> (pos % 8)) & 1
            codes[:, t] |= (v << bit).astype(np.uint8)
    return codes[:, :8], codes[:, 8:]


def _pack_q4_k(d, dmin, c, k, n):
    out = np.empty((d.shape[0], 144), np.uint8)
    out[:, 0:2] = _f16_bytes(d)
    out[:, 2:4] = _f16_bytes(dmin)
    out[:, 4:16] = _pack_scales(c, k)
    out[:, 16:144] = _pack_nibbles(n).reshape(-1, 128)
    return out


def _deq_q4_k(blk):
    d = _F(_f16_from_bytes(blk[:, 0:2]))
    dmin = _F(_f16_from_bytes(blk[:, 2:4]))
    c, k = _unpack_scales(blk[:, 4:16])
    S = d[:, None] * c.astype(_F32)                   # [n, 8]
    M = dmin[:, None] * k.astype(_F32)
    n = _unpack_nibbles(blk[:, 16:144].reshape(-1, 8, 16)).astype(_F32)   # [n, 8, 32]
    return (n * S[:, :, None] - M[:, :, None]).reshape(-1, 256)


# ---------------------------------------------------------------- public
def quantize(fmt: int, W: np.ndarray) -> np.ndarray:
    """W float32 [rows, cols] -> packed uint8 [rows, row_bytes(fmt, cols)]."""
    W = np.ascontiguousarray(W, dtype=_F32)
    if W.ndim == 1:
        W = W[None, :]
    W = W + _F32(0)                                   # reading 6: -0 -> +0
    rows, cols = W.shape
    rb = row_bytes(fmt, cols)
    if rb < 0:
        raise ValueError(f"cols={cols} is not a multiple of {BLOCK_WEIGHTS[fmt]}")
    if fmt == Q8_0:
        blk = _pack_q8_0(*_quant_q8_0(W.reshape(-1, 32)))
    elif fmt == Q4_0:
        blk = _pack_q4_0(*_quant_q4_0(W.reshape(-1, 32)))
    elif fmt == Q4_1:
        blk = _pack_q4_1(*_quant_q4_1(W.reshape(-1, 32)))
    elif fmt == Q4_K:
        blk = _pack_q4_k(*_quant_q4_k(W.reshape(-1, 8, 32)))
    else:
        raise ValueError(f"unknown format {fmt}")
    return blk.reshape(rows, rb)


def dequantize(fmt: int, packed: np.ndarray, cols: int) -> np.ndarray:
    """packed uint8 [rows, row_bytes] -> float32 [rows, cols]."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    rb = row_bytes(fmt, cols)
    rows = packed.size // rb
    blk = packed.reshape(-1, BLOCK_BYTES[fmt])
    if fmt == Q8_0:
        v = _deq_q8_0(blk)
    elif fmt == Q4_0:
        v = _deq_q4_0(blk)
    elif fmt == Q4_1:
        v = _deq_q4_1(blk)
    elif fmt == Q4_K:
        v = _deq_q4_k(blk)
    else:
        raise ValueError(f"unknown format {fmt}")
    return np.ascontiguousarray(v, dtype=_F32).reshape(rows, cols)


def quantize_dequantize(fmt: int, W: np.ndarray) -> np.ndarray:
    W = np.asarray(W, dtype=_F32)
    shape = W.shape
    W2 = W.reshape(-1, shape[-1])
    return dequantize(fmt, quantize(fmt, W2), W2.shape[1]).reshape(shape)
