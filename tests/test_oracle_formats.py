"""Pins for the format oracle against what the pages and the mathematics fix.

A plausible mistake in the oracle (a dropped term, a wrong sign, a wrong
index or nibble order, a missing clamp) fails at least one test here.
"""
import numpy as np
import pytest

import oracle
import synthetic
from oracle import Q8_0, Q4_0, Q4_1, Q4_K

NAME = {"Q8_0": Q8_0, "Q4_0": Q4_0, "Q4_1": Q4_1, "Q4_K": Q4_K}


def _hex(vals):
    return bytes(int(v, 16) for v in vals)


# ------------------------------------------------------------------ page numbers
def test_page2_bits_and_relative_errors(golden):
    """The handbook's printed table: bits/weight and relative error per format."""
    _, rows = golden("page2_formats.txt")
    w = synthetic.page2_sample().numpy().astype(np.float32)
    W = w.reshape(4096, 256)
    for name, bpw, rel in rows:
        fmt = NAME[name]
        assert oracle.bits_per_weight(fmt) == pytest.approx(float(bpw), abs=1e-12)
        deq = oracle.quantize_dequantize(fmt, W).reshape(-1).astype(np.float64)
        err = np.linalg.norm(deq - w) / np.linalg.norm(w.astype(np.float64))
        assert f"{err:.4f}" == rel, (name, err)


def test_studentt_generator_within_band():
    """Our own seeded Student-t sample (the bench's weights) lands within
    +-15 % of the page's relative errors (expected within ~1 %)."""
    w = synthetic.student_t((1024, 1024), seed=12345).numpy()
    page = {Q8_0: 0.0068, Q4_0: 0.1079, Q4_1: 0.0901, Q4_K: 0.0903}
    for fmt, ref in page.items():
        deq = oracle.quantize_dequantize(fmt, w).astype(np.float64)
        err = np.linalg.norm(deq - w) / np.linalg.norm(w.astype(np.float64))
        assert abs(err / ref - 1) < 0.05, (fmt, err)


def test_closed_form_bits_per_weight():
    # bits/weight = 8 * block bytes / block weights: (16 + 32*8)/32, (16+32*4)/32,
    # (32 + 32*4)/32, (2*16 + 16*6 + 256*4)/256
    assert oracle.bits_per_weight(Q8_0) == 8.5
    assert oracle.bits_per_weight(Q4_0) == 4.5
    assert oracle.bits_per_weight(Q4_1) == 5.0
    assert oracle.bits_per_weight(Q4_K) == 4.5


def test_epm_expert_bytes(golden):
    g, _ = golden("epq_expert_bytes.txt")
    weights, size = map(int, g["Q4_K"])
    assert weights == 3 * 512 * 2048
    packed = 2 * 512 * oracle.row_bytes(Q4_K, 2048) + 2048 * oracle.row_bytes(Q4_K, 512)
    assert packed == size


def test_row_bytes_rules():
    assert oracle.row_bytes(Q4_K, 4096) == 2304
    assert oracle.row_bytes(Q8_0, 4096) == 4352
    assert oracle.row_bytes(Q4_0, 14336) == 8064
    assert oracle.row_bytes(Q4_1, 256) == 160
    assert oracle.row_bytes(Q4_K, 100) == -1
    assert oracle.row_bytes(Q4_0, 48) == -1
    assert oracle.row_bytes(Q8_0, 0) == -1


# ------------------------------------------------------------------ hand blocks
def test_hand_block_q4_k(golden):
    g, _ = golden("hand_blocks.txt")
    c = [int(v) for v in g["q4k_values_c"]]
    k = [int(v) for v in g["q4k_values_k"]]
    n = list(range(16)) + list(range(15, -1, -1))
    x = np.array([[nn * (c[s] / 64) - k[s] / 128 for s in range(8) for nn in n]], np.float32)
    blk = oracle.quantize(Q4_K, x)[0].tobytes()
    assert blk[0:2] == _hex(g["q4k_d"])
    assert blk[2:4] == _hex(g["q4k_dmin"])
    assert blk[4:16] == _hex(g["q4k_scales"])
    for s in range(8):
        assert blk[16 + 16 * s:32 + 16 * s] == _hex(g["q4k_qs"]), s
    # every value is on the grid, so the round trip is exact
    assert np.array_equal(oracle.dequantize(Q4_K, np.frombuffer(blk, np.uint8)[None], 256), x)


def test_hand_block_q8_0(golden):
    g, _ = golden("hand_blocks.txt")
    q = [-127, -64, -1, 0] + list(range(1, 29))
    x = np.array([q], np.float32) / 16
    blk = oracle.quantize(Q8_0, x)[0].tobytes()
    assert blk[0:2] == _hex(g["q8_d"])
    assert blk[2:34] == _hex(g["q8_q"])


def test_hand_blocks_q4_0_tie_break(golden):
    g, _ = golden("hand_blocks.txt")
    base = np.array([((j % 16) - 8) / 4 for j in range(32)], np.float32)
    a = base.copy()
    a[5] = 2.0
    blk = oracle.quantize(Q4_0, a[None])[0].tobytes()
    assert blk[0:2] == _hex(g["q40a_d"]) and blk[2:] == _hex(g["q40a_qs"])
    b = base.copy()
    b[0], b[5] = 2.0, -2.0
    blk = oracle.quantize(Q4_0, b[None])[0].tobytes()
    assert blk[0:2] == _hex(g["q40b_d"]) and blk[2:] == _hex(g["q40b_qs"])


def test_hand_block_q4_1(golden):
    g, _ = golden("hand_blocks.txt")
    x = np.array([[-1 + (j % 16) / 4 for j in range(32)]], np.float32)
    blk = oracle.quantize(Q4_1, x)[0].tobytes()
    assert blk[0:2] == _hex(g["q41_d"])
    assert blk[2:4] == _hex(g["q41_m"])
    assert blk[4:20] == _hex(g["q41_qs"])


# ------------------------------------------------------------------ fp16 rounding
@pytest.mark.parametrize("value,bits", [
    (1.0 / 3.0, 0x3555),            # 0.333251953125
    (65504.0, 0x7BFF),              # largest finite
    (65520.0, 0x7C00),              # halfway to the next binade rounds up to inf
    (2.0 ** -24, 0x0001),           # smallest subnormal
    (2.0 ** -25, 0x0000),           # exact tie between 0 and 2^-24 -> even (0)
    (3 * 2.0 ** -25, 0x0002),       # tie between 1 and 2 ulps -> even (2)
    (1 + 2.0 ** -11, 0x3C00),       # tie -> even mantissa
    (1 + 3 * 2.0 ** -11, 0x3C02),   # tie -> even mantissa (up)
    (-0.25, 0xB400),
])
def test_fp16_round_to_nearest_even(value, bits):
    h = oracle.formats._f16(np.array([value], np.float32))
    assert int(h.view(np.uint16)[0]) == bits


# ------------------------------------------------------------------ degenerate blocks
def test_zero_blocks():
    z = np.zeros((1, 256), np.float32)
    assert oracle.quantize(Q8_0, z).tobytes() == bytes(8 * 34)
    assert oracle.quantize(Q4_1, z).tobytes() == bytes(8 * 20)
    # Q4_0: factor 0 / -8 = -0 (0x8000); codes 0 stored with the +8 offset
    q40 = oracle.quantize(Q4_0, z).reshape(8, 18)
    assert (q40[:, 0] == 0).all() and (q40[:, 1] == 0x80).all() and (q40[:, 2:] == 0x88).all()
    # Q4_K: d = dmin = +0, scale codes 1, min codes 0, nibbles 0
    q4k = oracle.quantize(Q4_K, z)[0]
    assert q4k[0:4].tobytes() == bytes(4)
    assert oracle.formats._unpack_scales(q4k[None, 4:16])[0].tolist() == [[1] * 8]
    assert q4k[16:].tobytes() == bytes(128)
    for fmt in oracle.FORMATS:
        assert not oracle.quantize_dequantize(fmt, z).any()
    # a negative zero input is the same block as +0
    for fmt in oracle.FORMATS:
        assert oracle.quantize(fmt, -z).tobytes() == oracle.quantize(fmt, z).tobytes()


def test_constant_blocks():
    v = np.float32(0.3)
    x = np.full((1, 256), v, np.float32)
    # Q4_1: range 0 -> d = 0, codes 0, dequant = fp16(min) exactly
    deq = oracle.quantize_dequantize(Q4_1, x)
    assert (deq == np.float32(np.float16(v))).all()
    # Q8_0 / Q4_0 reproduce a constant to within the fp16 factor
    assert np.allclose(oracle.quantize_dequantize(Q8_0, x), v, rtol=2e-3)
    assert np.allclose(oracle.quantize_dequantize(Q4_0, x), v, rtol=2e-3)
    # Q4_K, all positive: lo clamps to 0, so dmin = 0 and min codes are 0
    q = oracle.quantize(Q4_K, x)[0]
    assert q[2:4].tobytes() == bytes(2)
    assert oracle.formats._unpack_scales(q[None, 4:16])[1].tolist() == [[0] * 8]
    # negative constant: hi == lo -> every scale 0 -> d = 0 -> codes 1, nibbles 0,
    # and the block reconstructs to -dmin*k = the constant within fp16 x 6-bit error
    xn = -x
    qn = oracle.quantize(Q4_K, xn)[0]
    assert qn[0:2].tobytes() == bytes(2)
    assert np.allclose(oracle.quantize_dequantize(Q4_K, xn), -v, rtol=2e-2)


def test_all_positive_q4k_has_no_min():
    rng = np.random.default_rng(3)
    x = rng.uniform(0.01, 1.0, (4, 256)).astype(np.float32)
    q = oracle.quantize(Q4_K, x)
    for r in range(4):
        assert q[r, 2:4].tobytes() == bytes(2)
        assert (oracle.formats._unpack_scales(q[r:r + 1, 4:16])[1] == 0).all()


# ------------------------------------------------------------------ brute force
def _brute_codes(x, scale, offset, lo, hi):
    """Nearest grid index to x over all codes lo..hi, by exhaustive search.

    The grid value of code n is n*scale + offset; ties go to the even code
    (round half to even of the same division).
    """
    best = []
    for xv in x:
        t = np.float32(np.float32(xv - offset) / scale) if offset != 0 else np.float32(np.float32(xv) / scale)
        cands = list(range(lo, hi + 1))
        dist = [abs(float(t) - n) for n in cands]
        m = min(dist)
        ties = [n for n, d in zip(cands, dist) if d == m]
        best.append(ties[0] if len(ties) == 1 else [n for n in ties if n % 2 == 0][0])
    return best


def test_codes_are_nearest_grid_points():
    """Every stored code is the exhaustive-search nearest code for its scale."""
    rng = np.random.default_rng(7)
    x = (rng.standard_t(5, (8, 256)) * 0.02).astype(np.float32)
    F = oracle.formats._F
    # Q8_0
    p = oracle.quantize(Q8_0, x).reshape(-1, 34)
    for b in range(0, p.shape[0], 7):
        d = F(p[b, 0:2].view("<f2"))[0]
        q = p[b, 2:].view(np.int8).astype(int).tolist()
        assert q == _brute_codes(x.reshape(-1, 32)[b], d, 0, -127, 127)
        assert d == np.float32(np.float16(np.max(np.abs(x.reshape(-1, 32)[b])) / np.float32(127)))
    # Q4_0
    p = oracle.quantize(Q4_0, x).reshape(-1, 18)
    for b in range(0, p.shape[0], 7):
        d = F(p[b, 0:2].view("<f2"))[0]
        n = oracle.formats._unpack_nibbles(p[b:b + 1, 2:])[0].astype(int) - 8
        assert n.tolist() == _brute_codes(x.reshape(-1, 32)[b], d, 0, -8, 7)
    # Q4_1
    p = oracle.quantize(Q4_1, x).reshape(-1, 20)
    for b in range(0, p.shape[0], 7):
        d = F(p[b, 0:2].view("<f2"))[0]
        m = F(p[b, 2:4].view("<f2"))[0]
        n = oracle.formats._unpack_nibbles(p[b:b + 1, 4:])[0].astype(int)
        assert n.tolist() == _brute_codes(x.reshape(-1, 32)[b], d, m, 0, 15)
    # Q4_K: sub-block scale S = d*c, offset -M
    p = oracle.quantize(Q4_K, x).reshape(-1, 144)
    for b in range(p.shape[0]):
        d = F(p[b, 0:2].view("<f2"))[0]
        dmin = F(p[b, 2:4].view("<f2"))[0]
        c, k = oracle.formats._unpack_scales(p[b:b + 1, 4:16])
        xs = x.reshape(-1, 8, 32)[b]
        for s in range(8):
            S = np.float32(d * np.float32(c[0, s]))
            M = np.float32(dmin * np.float32(k[0, s]))
            n = oracle.formats._unpack_nibbles(p[b:b + 1, 16 + 16 * s:32 + 16 * s])[0].astype(int)
            # (x + M) / S == (x - (-M)) / S
            assert n.tolist() == _brute_codes(xs[s], S, -M, 0, 15), (b, s)
            # the 6-bit codes are the nearest codes of the sub-block scale and min
            lo = min(float(xs[s].min()), 0.0)
            sc = np.float32((np.float32(xs[s].max()) - np.float32(lo)) / np.float32(15))
            assert c[0, s] == _brute_codes([sc], d, 0, 1, 63)[0]
            assert k[0, s] == _brute_codes([np.float32(-lo)], dmin, 0, 0, 63)[0]


def test_dequant_single_rounding():
    """n*S - M (Q4_K) and n*d + m (Q4_1) round once: equal to the float64
    value rounded to float32."""
    rng = np.random.default_rng(11)
    x = (rng.standard_t(5, (4, 512)) * 0.02).astype(np.float32)
    F = oracle.formats._F
    p = oracle.quantize(Q4_K, x).reshape(-1, 144)
    deq = oracle.dequantize(Q4_K, p, 256)
    for b in range(p.shape[0]):
        d = float(F(p[b, 0:2].view("<f2"))[0])
        dmin = float(F(p[b, 2:4].view("<f2"))[0])
        c, k = oracle.formats._unpack_scales(p[b:b + 1, 4:16])
        n = oracle.formats._unpack_nibbles(p[b:b + 1, 16:].reshape(1, 8, 16))[0]
        ref = np.array([[n[s, j] * d * c[0, s] - dmin * k[0, s] for j in range(32)]
                        for s in range(8)], np.float64).reshape(-1).astype(np.float32)
        assert np.array_equal(deq[b], ref)
    p = oracle.quantize(Q4_1, x).reshape(-1, 20)
    deq = oracle.dequantize(Q4_1, p, 32)
    for b in range(0, p.shape[0], 5):
        d = float(F(p[b, 0:2].view("<f2"))[0])
        m = float(F(p[b, 2:4].view("<f2"))[0])
        n = oracle.formats._unpack_nibbles(p[b:b + 1, 4:])[0]
        ref = np.array([n[j] * d + m for j in range(32)]).astype(np.float32)
        assert np.array_equal(deq[b], ref)


def test_error_bound_per_weight():
    """Unclamped codes reconstruct within half a step of the input."""
    rng = np.random.default_rng(5)
    x = (rng.standard_t(5, (16, 256)) * 0.02).astype(np.float32)
    deq = oracle.quantize_dequantize(Q4_1, x).reshape(-1, 32)
    xb = x.reshape(-1, 32)
    step = (xb.max(1) - xb.min(1)) / 15
    # fp16 rounding of d and m adds at most a few ulps of fp16 times 15
    slack = 16 * 2.0 ** -11 * np.abs(xb).max(1)
    assert (np.abs(deq - xb) <= (step / 2 + slack)[:, None]).all()


PLANE_WIDTHS = {oracle.Q2_K: (64, 16, 4), oracle.Q6_K: (128, 64, 16, 2)}


def test_row_independence_and_block_order():
    """Packing row by row equals packing the matrix; blocks follow column order."""
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((3, 512))).astype(np.float32)
    for fmt in oracle.FORMATS:
        whole = oracle.quantize(fmt, x)
        for r in range(3):
            assert whole[r].tobytes() == oracle.quantize(fmt, x[r:r + 1])[0].tobytes()
        bw, bb = oracle.BLOCK_WEIGHTS[fmt], oracle.BLOCK_BYTES[fmt]
        singles = [oracle.quantize(fmt, x[0:1, blk * bw:(blk + 1) * bw])[0] for blk in range(512 // bw)]
        if fmt in PLANE_WIDTHS:
            # plane by plane: every plane holds the superblocks' entries in column order
            expected, o = [], 0
            for w in PLANE_WIDTHS[fmt]:
                expected += [sb[o:o + w] for sb in singles]
                o += w
            assert whole[0].tobytes() == np.concatenate(expected).tobytes()
        else:
            for blk, single in enumerate(singles):
                assert whole[0, blk * bb:(blk + 1) * bb].tobytes() == single.tobytes()
