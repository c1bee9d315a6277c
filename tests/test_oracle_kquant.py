"""Pins for the two 16-weight-sub-block K-quant formats of the format oracle
(Q2_K and Q6_K), independent of the oracle's own arithmetic:

* sizes: 84 and 210 bytes per 256 weights (2.625 and 6.5625 bits), the Q6_K
  size fixed by the per-expert byte count of "EPM ... 記憶體怎麼配置的";
* blocks built here by hand, byte by byte from the layout definition, decode
  to the values they were built from, and weights placed exactly on such a
  grid quantize back to those very bytes;
* on random blocks every stored weight code is a nearest grid point given
  the stored factors (brute force over all codes) and every sub-block scale
  code is the nearest multiple of the superblock factor;
* degenerate blocks (all zero, constant) and the reconstruction bounds.
"""
import numpy as np
import pytest

import oracle
import synthetic
from oracle import Q2_K, Q6_K

# the layout definition, restated: 2-bit field of sub-block position i
FIELD = [4, 8, 6, 10, 20, 24, 22, 26, 28, 0, 30, 2, 12, 16, 14, 18]


def _word_bytes(values):
    """16 two-bit values -> the 4 little-endian bytes of their sub-block word."""
    w = 0
    for i, v in enumerate(values):
        assert 0 <= v <= 3
        w |= int(v) << FIELD[i]
    return list(w.to_bytes(4, "little"))


def _f16le(v):
    return list(np.array([v], "<f2").view(np.uint8))


def test_sizes_and_bits_per_weight(golden):
    assert oracle.BLOCK_BYTES[Q2_K] == 84 and oracle.BLOCK_WEIGHTS[Q2_K] == 256
    assert oracle.bits_per_weight(Q2_K) == 2.625
    assert oracle.bits_per_weight(Q6_K) == 6.5625
    assert oracle.row_bytes(Q2_K, 4096) == 16 * 84
    assert oracle.row_bytes(Q6_K, 100) == -1
    g, _ = golden("epq_expert_bytes.txt")
    weights, size = map(int, g["Q4_K_gate_up+Q6_K_down"])
    assert weights == 3 * 512 * 2048
    assert 2 * 512 * oracle.row_bytes(oracle.Q4_K, 2048) + 2048 * oracle.row_bytes(Q6_K, 512) == size


def _q6k_hand(rng):
    """A Q6_K superblock on an exact grid: d = 2^-7, scale codes with
    max |c| = 127, each sub-block holding code -32 (its unique largest
    magnitude).  Returns (weights [256], expected bytes [210])."""
    d = 2.0 ** -7
    c = [127, -90, 64, -1, 3, 100, -127, 17, 45, -66, 2, 88, -5, 120, 9, -31]
    codes = rng.integers(-31, 32, size=(16, 16))
    for s in range(16):
        codes[s, (5 * s) % 16] = -32
    w = (codes * (d * np.array(c))[:, None]).reshape(256).astype(np.float32)
    u = (codes + 32).reshape(256)
    ql = [int(u[2 * b] & 15) | (int(u[2 * b + 1] & 15) << 4) for b in range(128)]
    qh = []
    for s in range(16):
        qh += _word_bytes([int(v) >> 4 for v in u[16 * s:16 * s + 16]])
    sc = [v & 0xFF for v in c]
    return w, np.array(ql + qh + sc + _f16le(d), np.uint8)


def _q2k_hand(rng):
    """A Q2_K superblock on an exact grid: d = 2^-6, dmin = 2^-5, step codes
    1..15 and lift codes 0..15 (each range's largest present), every
    sub-block holding codes 0 and 3."""
    d, dmin = 2.0 ** -6, 2.0 ** -5
    c = [15, 1, 7, 3, 9, 12, 2, 5, 11, 4, 6, 14, 8, 10, 13, 1]
    k = [0, 15, 3, 8, 1, 0, 12, 7, 2, 9, 4, 11, 6, 5, 14, 10]
    codes = rng.integers(0, 4, size=(16, 16))
    for s in range(16):
        codes[s, s] = 0
        codes[s, (s + 7) % 16] = 3
    w = (codes * (d * np.array(c))[:, None] - (dmin * np.array(k))[:, None]).reshape(256).astype(np.float32)
    cb = []
    for s in range(16):
        cb += _word_bytes(codes[s])
    sub = [c[s] | (k[s] << 4) for s in range(16)]
    return w, np.array(cb + sub + _f16le(d) + _f16le(dmin), np.uint8)


@pytest.mark.parametrize("fmt,maker", [(Q6_K, _q6k_hand), (Q2_K, _q2k_hand)])
def test_hand_block_round_trip(fmt, maker):
    rng = np.random.default_rng(fmt)
    w, expected = maker(rng)
    assert np.array_equal(oracle.dequantize(fmt, expected[None, :], 256)[0], w)
    assert np.array_equal(oracle.quantize(fmt, w[None, :])[0], expected)


def test_hand_blocks_in_a_planar_row():
    """Three superblocks in one row: each plane holds the three entries in
    superblock order (codes of all three, then scales of all three, ...)."""
    rng = np.random.default_rng(7)
    blocks = [_q6k_hand(rng) for _ in range(3)]
    w = np.concatenate([b[0] for b in blocks])[None, :]
    planes = [(0, 128), (128, 192), (192, 208), (208, 210)]
    row = np.concatenate([b[1][lo:hi] for lo, hi in planes for b in blocks])
    assert np.array_equal(oracle.quantize(Q6_K, w)[0], row)
    assert np.array_equal(oracle.dequantize(Q6_K, row[None, :], 768), w)


def _fields(word_bytes):
    w = int.from_bytes(bytes(word_bytes), "little")
    return [(w >> FIELD[i]) & 3 for i in range(16)]


def _unpack_q2k(blk):
    codes = np.array([_fields(blk[4 * s:4 * s + 4]) for s in range(16)])
    c = blk[64:80] & 15
    k = blk[64:80] >> 4
    d, dmin = blk[80:82].view("<f2")[0], blk[82:84].view("<f2")[0]
    return codes, c, k, float(d), float(dmin)


def _unpack_q6k(blk):
    lo = np.array([(blk[j >> 1] >> (4 * (j & 1))) & 15 for j in range(256)]).reshape(16, 16)
    hi = np.array([_fields(blk[128 + 4 * s:132 + 4 * s]) for s in range(16)])
    c = blk[192:208].view(np.int8).astype(np.int64)
    d = float(blk[208:210].view("<f2")[0])
    return (lo | (hi << 4)) - 32, c, d


def test_q2k_codes_are_nearest_given_stored_factors():
    W = synthetic.student_t((6, 256), seed=3).numpy()
    packed = oracle.quantize(Q2_K, W)
    for r in range(6):
        codes, c, k, d, dmin = _unpack_q2k(packed[r])
        w = W[r].reshape(16, 16).astype(np.float64)
        lo = np.minimum(w.min(1), 0.0)
        step, lift = (w.max(1) - lo) / 3, -lo
        assert d == np.float16(np.float32(step.max() / 15)) and dmin == np.float16(np.float32(lift.max() / 15))
        for s in range(16):
            # scale codes: nearest multiple of the stored factor within 1..15 / 0..15
            assert abs(step[s] - c[s] * d) <= min(abs(step[s] - cc * d) for cc in range(1, 16)) + 1e-6 * d
            assert abs(lift[s] - k[s] * dmin) <= min(abs(lift[s] - kk * dmin) for kk in range(16)) + 1e-6 * dmin
            S, M = c[s] * d, k[s] * dmin
            for j in range(16):
                err = abs(w[s, j] - (codes[s, j] * S - M))
                assert err <= min(abs(w[s, j] - (n * S - M)) for n in range(4)) + 1e-6 * S


def test_q6k_codes_are_nearest_given_stored_factors():
    W = synthetic.student_t((6, 256), seed=4).numpy()
    packed = oracle.quantize(Q6_K, W)
    for r in range(6):
        n, c, d = _unpack_q6k(packed[r])
        w = W[r].reshape(16, 16).astype(np.float64)
        peak = w[np.arange(16), np.abs(w).argmax(1)]
        scale = peak / -32
        assert d == np.float16(np.float32(np.abs(scale).max() / 127))
        for s in range(16):
            assert abs(scale[s] - c[s] * d) <= min(abs(scale[s] - cc * d) for cc in range(-127, 128)) + 1e-6 * d
            S = c[s] * d
            for j in range(16):
                err = abs(w[s, j] - n[s, j] * S)
                assert err <= min(abs(w[s, j] - m * S) for m in range(-32, 32)) + 1e-6 * abs(S)


def test_degenerate_blocks():
    z = np.zeros((1, 256), np.float32)
    p2 = oracle.quantize(Q2_K, z)[0]
    assert (p2[:64] == 0).all() and (p2[64:80] == 1).all() and (p2[80:] == 0).all()
    p6 = oracle.quantize(Q6_K, z)[0]
    assert (p6[:128] == 0).all() and (p6[192:] == 0).all()
    assert _unpack_q6k(p6)[0].tolist() == [[0] * 16] * 16        # u = 32: code 0
    for fmt in (Q2_K, Q6_K):
        assert not oracle.dequantize(fmt, oracle.quantize(fmt, z), 256).any()
    # a constant positive superblock: every weight decodes within half a step
    cst = np.full((1, 256), 0.25, np.float32)
    for fmt in (Q2_K, Q6_K):
        back = oracle.dequantize(fmt, oracle.quantize(fmt, cst), 256)
        assert np.abs(back - cst).max() <= 0.25 / 3


def test_reconstruction_bounds():
    """Error bounds from the arithmetic.  Q2_K: a stored step S is within d
    of the ideal step st (half a factor by rounding, a full one where the
    code clamps up to 1) and a stored lift within dmin/2 of the ideal one,
    so a grid level n*S - M (n <= 3) is within 3d + dmin/2 of the ideal level
    and each weight within st/2 + 3d + dmin/2.  Q6_K: the stored scale is
    within d/2 of the ideal one, the 64 levels m*S (|m| <= 32) within 16 d,
    and each weight within |scale| (half a step, a full step where the code
    clamps at 31) + 16 d."""
    W = synthetic.student_t((32, 1024), seed=9).numpy()
    back = oracle.dequantize(Q2_K, oracle.quantize(Q2_K, W), 1024).reshape(-1, 16, 16).astype(np.float64)
    w = W.reshape(-1, 16, 16).astype(np.float64)
    lo = np.minimum(w.min(2), 0)
    st, lift = (w.max(2) - lo) / 3, -lo
    d, dmin = st.max(1, keepdims=True) / 15, lift.max(1, keepdims=True) / 15
    bound = st / 2 + 3 * d + dmin / 2
    assert (np.abs(back - w).max(2) <= bound * (1 + 1e-3) + 1e-12).all()
    back = oracle.dequantize(Q6_K, oracle.quantize(Q6_K, W), 1024).reshape(-1, 16, 16).astype(np.float64)
    scale = np.abs(w).max(2) / 32
    d = scale.max(1, keepdims=True) / 127
    bound = scale + 16 * d
    assert (np.abs(back - w).max(2) <= bound * (1 + 1e-3) + 1e-12).all()
