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

Two more K-quant formats that the pages name without defining them -- Q2_K
(the 2-bit experts of "smolmaxxing" and the 2-bit experts of "Flash-MoE")
and Q6_K (the down projections of "EPM ... 記憶體怎麼配置的", 2,039,808 B per
expert, i.e. 210 B per 256 weights) -- follow the same two-level idea at
the sizes those pages fix:

* Q2_K: superblocks of 256 = 16 sub-blocks of 16 weights; per sub-block an
  affine grid of 4 levels (step = range over 3 from min(min, 0), lift =
  -that floor), steps and lifts coded as 4-bit multiples of two fp16
  factors (largest / 15); 2-bit codes.  84 B per superblock (2.625 bits).
* Q6_K: superblocks of 256 = 16 sub-blocks of 16; symmetric like Q4_0: the
  sub-block scale is its signed largest-magnitude weight over -32 (that
  weight lands on code -32), coded as an int8 multiple of one fp16 factor
  (largest |scale| / 127); 6-bit codes -32..31.  210 B per superblock
  (6.5625 bits).  A Q6_K weight is exact in float32 (18 x 6 bits).

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
   Q2_K and Q6_K rows are stored plane by plane (every plane's entries stay
   aligned to their own size for wide loads), for a row of nsb superblocks:
     Q2_K  codes[64 nsb] | sub-block codes[16 nsb] | f16 (d, dmin)[nsb]
           sub-block s of a superblock owns the little-endian 32-bit word
           s of its 64 code bytes; sub-block code byte = c | k << 4
     Q6_K  low nibbles[128 nsb] | high bits[64 nsb] | int8 scale codes[16 nsb]
           | f16 d[nsb]; u = code + 32 in 0..63: u & 15 of superblock
           weight j in byte j>>1 of its 128 (low nibble when j is even);
           u >> 4 of sub-block s in word s of its 64 high-bit bytes
   A 2-bit field (a Q2_K code, a Q6_K high part) of position i = 0..15 of a
   sub-block starts at bit FIELD[i] of the sub-block's word, FIELD = (4, 8,
   6, 10, 20, 24, 22, 26, 28, 0, 30, 2, 12, 16, 14, 18): an order that lets
   a decoder reach two fields at a time in fp16 mantissa position with one
   mask, after at most one shift and one rotation of the word.
6. Signed zeros: inputs are first mapped ``x -> x + 0`` (so -0 becomes +0)
   and the Q4_K min is formed as ``0 - lo``; every max/min then has one
   well-defined result and a zero factor is always +0 (Q4_0's factor of an
   all-zero block is +0 / -8 = -0, kept as the division gives it).
   Inputs must be finite.
"""
from __future__ import annotations

import numpy as np

Q8_0, Q4_0, Q4_1, Q4_K, Q2_K, Q6_K = 0, 1, 2, 3, 4, 5
FORMATS = (Q8_0, Q4_0, Q4_1, Q4_K, Q2_K, Q6_K)
NAMES = {Q8_0: "Q8_0", Q4_0: "Q4_0", Q4_1: "Q4_1", Q4_K: "Q4_K", Q2_K: "Q2_K", Q6_K: "Q6_K"}
BLOCK_WEIGHTS = {Q8_0: 32, Q4_0: 32, Q4_1: 32, Q4_K: 256, Q2_K: 256, Q6_K: 256}
BLOCK_BYTES = {Q8_0: 34, Q4_0: 18, Q4_1: 20, Q4_K: 144, Q2_K: 84, Q6_K: 210}

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


def _encode_q2_k(sbs: np.ndarray):
    """Superblocks [nsb, 16, 16] -> planes (codes [nsb, 64], sub-block codes
    [nsb, 16], factors [nsb, 4])."""
    floor = np.minimum(np.min(sbs, axis=2), _F32(0))
    sub_step = (np.max(sbs, axis=2) - floor) / _F32(3.0)
    sub_lift = _F32(0) - floor
    d = _f16(np.max(sub_step, axis=1) / _F32(15.0))
    dmin = _f16(np.max(sub_lift, axis=1) / _F32(15.0))
    dF, dminF = _F(d)[:, None], _F(dmin)[:, None]
    c = np.where(dF == 0, _F32(1), _nearest_codes(sub_step, dF, _F32(0), 1, 15))
    k = _nearest_codes(sub_lift, dminF, _F32(0), 0, 15)
    step = dF * c           # exact: 11 x 4 significant bits
    lift = dminF * k        # exact
    n = _nearest_codes(sbs, step[:, :, None], lift[:, :, None], 0, 3)
    codes = _fields_to_words(n).reshape(-1, 64)
    sub = (c.astype(np.uint8) | (k.astype(np.uint8) << 4)).astype(np.uint8)
    fac = np.concatenate([_f16_bytes(d), _f16_bytes(dmin)], axis=1)
    return codes, sub, fac


def _encode_q6_k(sbs: np.ndarray):
    """Superblocks [nsb, 16, 16] -> planes (low nibbles [nsb, 128], high bits
    [nsb, 64], scale codes [nsb, 16], factor [nsb, 2])."""
    first_peak = np.argmax(np.abs(sbs), axis=2)
    signed_peak = np.take_along_axis(sbs, first_peak[:, :, None], axis=2)[:, :, 0]
    sub_scale = signed_peak / _F32(-32.0)
    d = _f16(np.max(np.abs(sub_scale), axis=1) / _F32(127.0))
    dF = _F(d)[:, None]
    c = _nearest_codes(sub_scale, dF, _F32(0), -127, 127)
    step = dF * c           # exact: 11 x 7 significant bits
    n = _nearest_codes(sbs, step[:, :, None], _F32(0), -32, 31)
    u = (n + _F32(32)).astype(np.uint8).reshape(-1, 256)
    ql = (u[:, 0::2] & 15) | ((u[:, 1::2] & 15) << 4)
    qh = _fields_to_words((u >> 4).reshape(-1, 16, 16)).reshape(-1, 64)
    return ql.astype(np.uint8), qh, c.astype(np.int8).view(np.uint8), _f16_bytes(d)


FIELD = (4, 8, 6, 10, 20, 24, 22, 26, 28, 0, 30, 2, 12, 16, 14, 18)


def _fields_to_words(f: np.ndarray) -> np.ndarray:
    """2-bit values [n, 16 sub-blocks, 16 positions] -> [n, 16 * 4] bytes:
    one little-endian word per sub-block, position i at bit FIELD[i]."""
    f = np.asarray(f).astype(np.uint32)
    words = np.zeros(f.shape[:2], np.uint32)
    for i, b in enumerate(FIELD):
        words |= f[:, :, i] << np.uint32(b)
    return np.ascontiguousarray(words.astype("<u4")).view(np.uint8).reshape(f.shape[0], -1)


def _words_to_fields(b: np.ndarray) -> np.ndarray:
    """Inverse of _fields_to_words: [n, 64] bytes -> [n, 16, 16] values."""
    words = np.ascontiguousarray(b).view("<u4").reshape(b.shape[0], 16).astype(np.uint32)
    return np.stack([(words >> np.uint32(FIELD[i])) & np.uint32(3) for i in range(16)], axis=2)


def _rows_from_planes(planes, rows: int):
    """Per-superblock planes [rows * nsb, w] -> rows of consecutive planes."""
    return np.concatenate([p.reshape(rows, -1) for p in planes], axis=1)


def _planes_of_rows(packed: np.ndarray, nsb: int, widths):
    """Inverse of _rows_from_planes: [rows, sum(w) * nsb] -> [rows * nsb, w] each."""
    out, o = [], 0
    for w in widths:
        out.append(np.ascontiguousarray(packed[:, o:o + w * nsb]).reshape(-1, w))
        o += w * nsb
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


def _decode_q2_k(codes, sub, fac):
    d = _F(_f16_from_bytes(fac[:, 0:2]))
    dmin = _F(_f16_from_bytes(fac[:, 2:4]))
    c = (sub & 15).astype(_F32)
    k = (sub >> 4).astype(_F32)
    step = d[:, None] * c                              # [n, 16]
    lift = dmin[:, None] * k
    n = _words_to_fields(codes).astype(_F32)
    return (n * step[:, :, None] - lift[:, :, None]).reshape(-1, 256)


def _decode_q6_k(ql, qh, sc, dbytes):
    d = _F(_f16_from_bytes(dbytes))
    c = sc.view(np.int8).astype(_F32)
    step = d[:, None] * c
    lo = np.empty((ql.shape[0], 256), np.uint8)
    lo[:, 0::2] = ql & 15
    lo[:, 1::2] = ql >> 4
    hi = _words_to_fields(qh).reshape(-1, 256).astype(np.uint8)
    n = (lo | (hi << 4)).astype(_F32) - _F32(32)
    return (n.reshape(-1, 16, 16) * step[:, :, None]).reshape(-1, 256)


_PLANES = {Q2_K: (_encode_q2_k, _decode_q2_k, (64, 16, 4)), Q6_K: (_encode_q6_k, _decode_q6_k, (128, 64, 16, 2))}

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
    if fmt not in _ENCODERS and fmt not in _PLANES:
        raise ValueError(f"unknown format {fmt}")
    if rb < 0:
        raise ValueError(f"cols={cols} is not a multiple of {BLOCK_WEIGHTS[fmt]}")
    if fmt in _PLANES:
        return _rows_from_planes(_PLANES[fmt][0](W.reshape(-1, 16, 16)), rows)
    encode, run_shape = _ENCODERS[fmt]
    return encode(W.reshape(run_shape)).reshape(rows, rb)


def dequantize(fmt: int, packed: np.ndarray, cols: int) -> np.ndarray:
    """packed uint8 [rows, row_bytes] -> float32 [rows, cols]."""
    if fmt not in _DECODERS and fmt not in _PLANES:
        raise ValueError(f"unknown format {fmt}")
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    rb = row_bytes(fmt, cols)
    rows = packed.size // rb
    if fmt in _PLANES:
        _, decode, widths = _PLANES[fmt]
        v = decode(*_planes_of_rows(packed.reshape(rows, rb), cols // 256, widths))
        return np.ascontiguousarray(v, dtype=_F32).reshape(rows, cols)
    v = _DECODERS[fmt](packed.reshape(-1, BLOCK_BYTES[fmt]))
    return np.ascontiguousarray(v, dtype=_F32).reshape(rows, cols)


def quantize_dequantize(fmt: int, W: np.ndarray) -> np.ndarray:
    W = np.asarray(W, dtype=_F32)
    shape = W.shape
    W2 = W.reshape(-1, shape[-1])
    return dequantize(fmt, quantize(fmt, W2), W2.shape[1]).reshape(shape)
