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


def _nearest_codes(w: np.ndarray, step: np.ndarray, offset, lo: int, hi: int) -> np.ndarray:
    """Codes of an affine grid, in float32: the integer nearest to
    (w + offset) / step (ties to even), clamped to [lo, hi]; 0 wherever the
    step is 0 (reading 3)."""
    w = np.asarray(w, _F32)
    step = np.asarray(step, _F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (w + np.asarray(offset, _F32)) / step
    code = np.clip(np.rint(t), _F32(lo), _F32(hi))
    return np.where(step == 0, _F32(0), code)


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


# ---------------------------------------------------------------- encoders
# Every format codes a run of weights on an affine grid w ~ step * n - offset
# with small integers n; the formats differ in how the grid of a run is
# chosen and stored.  Each encoder takes runs [nb, run] (float32, -0 already
# mapped to +0) and returns the packed bytes [nb, block_bytes].

def _encode_q8_0(runs: np.ndarray) -> np.ndarray:
    """Symmetric grid through 0 whose step puts the largest |w| at 127."""
    step = _f16(np.max(np.abs(runs), axis=1) / _F32(127.0))
    n = _nearest_codes(runs, _F(step)[:, None], _F32(0), -127, 127)
    out = np.empty((runs.shape[0], 34), np.uint8)
    out[:, 0:2] = _f16_bytes(step)
    out[:, 2:34] = n.astype(np.int8).view(np.uint8)
    return out


def _encode_q4_0(runs: np.ndarray) -> np.ndarray:
    """Symmetric grid whose step is the signed weight of largest magnitude
    (first such index) over -8, so that this weight sits on code -8; codes
    -8..7 are stored with an offset of 8."""
    first_peak = np.argmax(np.abs(runs), axis=1)
    signed_peak = np.take_along_axis(runs, first_peak[:, None], axis=1)[:, 0]
    step = _f16(signed_peak / _F32(-8.0))
    n = _nearest_codes(runs, _F(step)[:, None], _F32(0), -8, 7)
    out = np.empty((runs.shape[0], 18), np.uint8)
    out[:, 0:2] = _f16_bytes(step)
    out[:, 2:18] = _pack_nibbles(n + _F32(8))
    return out


def _encode_q4_1(runs: np.ndarray) -> np.ndarray:
    """Grid from the run's minimum m (stored) with step (max - min) / 15."""
    lowest, highest = np.min(runs, axis=1), np.max(runs, axis=1)
    step = _f16((highest - lowest) / _F32(15.0))
    base = _f16(lowest)
    n = _nearest_codes(runs, _F(step)[:, None], -_F(base)[:, None], 0, 15)
    out = np.empty((runs.shape[0], 20), np.uint8)
    out[:, 0:2] = _f16_bytes(step)
    out[:, 2:4] = _f16_bytes(base)
    out[:, 4:20] = _pack_nibbles(n)
    return out


def _encode_q4_k(sbs: np.ndarray) -> np.ndarray:
    """Two-level grid over superblocks [nsb, 8, 32].  Each sub-block's grid
    starts at floor = min(its minimum, 0) and spans its range in 15 steps;
    the eight steps are coded as 6-bit multiples (1..63) of one fp16 factor
    d = largest step / 63, the eight lifts -floor as 6-bit multiples (0..63)
    of dmin = largest lift / 63; weights are then coded on the sub-block's
    stored grid (step c*d, lift k*dmin)."""
    floor = np.minimum(np.min(sbs, axis=2), _F32(0))
    sub_step = (np.max(sbs, axis=2) - floor) / _F32(15.0)
    sub_lift = _F32(0) - floor
    d = _f16(np.max(sub_step, axis=1) / _F32(63.0))
    dmin = _f16(np.max(sub_lift, axis=1) / _F32(63.0))
    dF, dminF = _F(d)[:, None], _F(dmin)[:, None]
    c = np.where(dF == 0, _F32(1), _nearest_codes(sub_step, dF, _F32(0), 1, 63))
    k = _nearest_codes(sub_lift, dminF, _F32(0), 0, 63)
    step = dF * c           # exact: 11 x 6 significant bits
    lift = dminF * k        # exact
    n = _nearest_codes(sbs, step[:, :, None], lift[:, :, None], 0, 15)
    out = np.empty((sbs.shape[0], 144), np.uint8)
    out[:, 0:2] = _f16_bytes(d)
    out[:, 2:4] = _f16_bytes(dmin)
    out[:, 4:16] = _pack_scales(c.astype(np.uint8), k.astype(np.uint8))
    out[:, 16:144] = _pack_nibbles(n).reshape(-1, 128)
    return out


# ---------------------------------------------------------------- decoders
# w = step * n - offset with one rounding (step * n is exact in float32).

def _decode_q8_0(blk):
    step = _F(_f16_from_bytes(blk[:, 0:2]))
    n = np.ascontiguousarray(blk[:, 2:34]).view(np.int8).astype(_F32)
    return step[:, None] * n


def _decode_q4_0(blk):
    step = _F(_f16_from_bytes(blk[:, 0:2]))
    n = _unpack_nibbles(blk[:, 2:18]).astype(_F32) - _F32(8)
    return step[:, None] * n


def _decode_q4_1(blk):
    step = _F(_f16_from_bytes(blk[:, 0:2]))
    base = _F(_f16_from_bytes(blk[:, 2:4]))
    n = _unpack_nibbles(blk[:, 4:20]).astype(_F32)
    return n * step[:, None] + base[:, None]


def _decode_q4_k(blk):
    d = _F(_f16_from_bytes(blk[:, 0:2]))
    dmin = _F(_f16_from_bytes(blk[:, 2:4]))
    c, k = _unpack_scales(blk[:, 4:16])
    step = d[:, None] * c.astype(_F32)                 # [n, 8]
    lift = dmin[:, None] * k.astype(_F32)
    n = _unpack_nibbles(blk[:, 16:144].reshape(-1, 8, 16)).astype(_F32)   # [n, 8, 32]
    return (n * step[:, :, None] - lift[:, :, None]).reshape(-1, 256)


_ENCODERS = {Q8_0: (_encode_q8_0, (-1, 32)), Q4_0: (_encode_q4_0, (-1, 32)),
             Q4_1: (_encode_q4_1, (-1, 32)), Q4_K: (_encode_q4_k, (-1, 8, 32))}
_DECODERS = {Q8_0: _decode_q8_0, Q4_0: _decode_q4_0, Q4_1: _decode_q4_1, Q4_K: _decode_q4_k}


# ---------------------------------------------------------------- public
def quantize(fmt: int, W: np.ndarray) -> np.ndarray:
    """W float32 [rows, cols] -> packed uint8 [rows, row_bytes(fmt, cols)]."""
    W = np.ascontiguousarray(W, dtype=_F32)
    if W.ndim == 1:
        W = W[None, :]
    W = W + _F32(0)                                   # reading 6: -0 -> +0
    rows, cols = W.shape
    rb = row_bytes(fmt, cols)
    if fmt not in _ENCODERS:
        raise ValueError(f"unknown format {fmt}")
    if rb < 0:
        raise ValueError(f"cols={cols} is not a multiple of {BLOCK_WEIGHTS[fmt]}")
    encode, run_shape = _ENCODERS[fmt]
    return encode(W.reshape(run_shape)).reshape(rows, rb)


def dequantize(fmt: int, packed: np.ndarray, cols: int) -> np.ndarray:
    """packed uint8 [rows, row_bytes] -> float32 [rows, cols]."""
    if fmt not in _DECODERS:
        raise ValueError(f"unknown format {fmt}")
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    rb = row_bytes(fmt, cols)
    rows = packed.size // rb
    v = _DECODERS[fmt](packed.reshape(-1, BLOCK_BYTES[fmt]))
    return np.ascontiguousarray(v, dtype=_F32).reshape(rows, cols)


def quantize_dequantize(fmt: int, W: np.ndarray) -> np.ndarray:
    W = np.asarray(W, dtype=_F32)
    shape = W.shape
    W2 = W.reshape(-1, shape[-1])
    return dequantize(fmt, quantize(fmt, W2), W2.shape[1]).reshape(shape)
