"""CPU model of the CUDA-core dequant-GEMV engine's arithmetic, checked
against the float64 oracle (host logic; no GPU).

The engine (Q8_0 / Q4_0 / Q4_1, and Q4_K under the CUDA-core engine) never
converts a code to float with an instruction: a packed word masked to one
code, read as an IEEE float32 bit pattern, is the exact value
code * 2^(shift - 149) (a subnormal or the smallest normals, where the
encoding is linear), shift being the code's bit position after the two
nibbles above bit 23 (or the top byte) are moved down by 16.  Each
activation is stored as x * 2^(126 - E - shift) (|x| < 2^E for the whole
vector), so every product is code * x * 2^(-23 - E); per 32-weight column
the format's scale, offset and minimum enter once, with the column's sum of
x in the same units, and the row total is scaled back by 2^(23 + E).

The model below builds those patterns from the packed bytes (read here
directly, not through the oracle's decoder), takes the products and sums
in float64 and must match oracle.gemv_f64 within 1e-9 of sum |w x|: the
algebra is exact, so only float64 rounding remains.  A wrong shift, mask
or offset misses by orders of magnitude.
"""
import numpy as np
import pytest

import oracle
import synthetic

Q8_0, Q4_0, Q4_1, Q4_K = oracle.Q8_0, oracle.Q4_0, oracle.Q4_1, oracle.Q4_K

# Bit position each weight of a 32-weight column carries in its pattern.
SHIFT_NIBBLE = [4 * (j & 7) if (j & 7) < 6 else 4 * ((j & 7) - 4) for j in range(32)]
SHIFT_BYTE = [8 if (j & 3) == 3 else 8 * (j & 3) for j in range(32)]
Q8_BIAS = 128
Q4_0_OFFSET = 8


def _pattern(u: int) -> float:
    """uint32 bit pattern -> its float32 value (exact)."""
    return float(np.array([u], np.uint32).view(np.float32)[0])


def _f16(b: bytes) -> float:
    return float(np.frombuffer(b, np.float16)[0])


def _words(b: bytes):
    return [int.from_bytes(b[4 * i:4 * i + 4], "little") for i in range(len(b) // 4)]


def _bound_exponent(amax: float) -> int:
    eb = int(np.array([amax], np.float32).view(np.uint32)[0] >> 23) & 0xFF
    return max(eb, 1) - 126


def _nibble_sum(words, scaled):
    """sum over 4 words of 8 nibbles: pattern (masked, the top two moved
    down by 16) times the scaled activation of the same weight."""
    acc = 0.0
    for i, w in enumerate(words):
        h = w >> 16
        pats = [w & 0xF, w & 0xF0, w & 0xF00, w & 0xF000, w & 0xF0000, w & 0xF00000, h & 0xF00, h & 0xF000]
        for p in range(8):
            acc += _pattern(pats[p]) * scaled[8 * i + p]
    return acc


def _byte_sum(words, scaled):
    """sum over 8 words of 4 int8 codes, each biased by the XOR with 0x80."""
    acc = 0.0
    for i, w in enumerate(words):
        u = w ^ 0x80808080
        pats = [u & 0xFF, u & 0xFF00, u & 0xFF0000, (u >> 16) & 0xFF00]
        for p in range(4):
            acc += _pattern(pats[p]) * scaled[4 * i + p]
    return acc


def _row(fmt, row: bytes, x: np.ndarray, E: int) -> float:
    cols = x.size
    shift = SHIFT_BYTE if fmt == Q8_0 else SHIFT_NIBBLE
    total = 0.0
    for c in range(cols // 32):
        xc = x[32 * c:32 * c + 32].astype(np.float64)
        scaled = [xc[j] * 2.0 ** (126 - E - shift[j]) for j in range(32)]
        xs = float(np.sum(xc)) * 2.0 ** (-23 - E)
        if fmt == Q8_0:
            blk = row[34 * c:34 * c + 34]
            part = _f16(blk[0:2]) * (_byte_sum(_words(blk[2:34]), scaled) - Q8_BIAS * xs)
        elif fmt == Q4_0:
            blk = row[18 * c:18 * c + 18]
            part = _f16(blk[0:2]) * (_nibble_sum(_words(blk[2:18]), scaled) - Q4_0_OFFSET * xs)
        elif fmt == Q4_1:
            blk = row[20 * c:20 * c + 20]
            part = _f16(blk[0:2]) * _nibble_sum(_words(blk[4:20]), scaled) + _f16(blk[2:4]) * xs
        else:  # Q4_K: column c is sub-block s of superblock sb
            sb, s = c >> 3, c & 7
            blk = row[144 * sb:144 * sb + 144]
            stream = int.from_bytes(blk[4:16], "little")
            code, mcode = (stream >> (6 * s)) & 63, (stream >> (48 + 6 * s)) & 63
            S, M = _f16(blk[0:2]) * code, _f16(blk[2:4]) * mcode
            part = S * _nibble_sum(_words(blk[16 + 16 * s:32 + 16 * s]), scaled) - M * xs
        total += part
    return total * 2.0 ** (23 + E)


def _model(fmt, packed, x):
    rows = packed.shape[0]
    out = np.zeros((x.shape[0], rows))
    for v in range(x.shape[0]):
        E = _bound_exponent(float(np.max(np.abs(x[v]))))
        for r in range(rows):
            out[v, r] = _row(fmt, bytes(packed[r]), x[v], E)
    return out


def _case(fmt, seed, cols, scale):
    W = synthetic.student_t((4, cols), seed=seed).numpy()
    packed = oracle.quantize(fmt, W)
    x = (synthetic.normal((2, cols), seed=seed + 1).numpy() * np.float32(scale)).astype(np.float32)
    return packed, x


@pytest.mark.parametrize("fmt", [Q8_0, Q4_0, Q4_1, Q4_K])
@pytest.mark.parametrize("scale", [1.0, 1e-6, 3e5])
def test_column_engine_model_matches_oracle(fmt, scale):
    packed, x = _case(fmt, 30 + fmt, 512, scale)
    got = _model(fmt, packed, x)
    ref = oracle.gemv_f64(fmt, packed, x, 512)
    bound = oracle.gemv_bound(fmt, packed, x, 512)
    assert (np.abs(got - ref) <= 1e-9 * bound + 1e-300).all(), (np.abs(got - ref) / bound).max()


def test_column_engine_model_catches_planted_slips():
    """Not vacuous: the top nibbles left at their own bit positions, or a
    Q8_0 bias of 127, each miss by far more than the bound."""
    global SHIFT_NIBBLE, Q8_BIAS
    packed, x = _case(Q4_0, 41, 256, 1.0)
    ref = oracle.gemv_f64(Q4_0, packed, x, 256)
    bound = oracle.gemv_bound(Q4_0, packed, x, 256)
    saved = SHIFT_NIBBLE
    try:
        SHIFT_NIBBLE = [4 * (j & 7) for j in range(32)]
        bad = _model(Q4_0, packed, x)
    finally:
        SHIFT_NIBBLE = saved
    assert (np.abs(bad - ref) > 1e-3 * bound).any()
    packed, x = _case(Q8_0, 43, 256, 1.0)
    ref = oracle.gemv_f64(Q8_0, packed, x, 256)
    bound = oracle.gemv_bound(Q8_0, packed, x, 256)
    try:
        Q8_BIAS = 127
        bad = _model(Q8_0, packed, x)
    finally:
        Q8_BIAS = 128
    assert (np.abs(bad - ref) > 1e-3 * bound).any()
