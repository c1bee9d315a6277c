"""CPU models of the two Q4_K tensor-core operand layouts, checked against the
float64 oracle (host logic; no GPU).

Both engines feed `mma.sync.m16n8k16` (fp16 A and B, fp32 C) with the
fragment layout of the PTX ISA: lane (g, t) = (lane / 4, lane % 4) holds
A[g][2t, 2t+1], A[g+8][2t, 2t+1], A[g][2t+8, 2t+9], A[g+8][2t+8, 2t+9] in its
four A registers, B[2t, 2t+1][g] and B[2t+8, 2t+9][g] in its two B
registers, and C[g][2t], C[g][2t+1], C[g+8][2t], C[g+8][2t+1].  The models
below build every register from the packed bytes and from x exactly as the
kernels' comments state, multiply with that fragment map (exact float64
products and sums), apply the kernels' epilogues and compare with
oracle.gemv_f64 within 1e-6 of sum |w x| (the fp16 hi + lo split of x leaves
~2^-22 of each term).  A wrong mask, shift, scale power, slot or sum here
fails by orders of magnitude.

* block-diagonal engine (one vector): the 8 B columns are (owner t', hi/lo),
  zero outside the owner's k-slots; class-B codes carry 16x, their x slots
  2^-4 x; sub-block scale and min applied in float32 per owner after the
  MMAs.
* vector-column engine (2..8 vectors): the 8 B columns are vectors; one
  HMUL2 folds the sub-block scale into the code operand (c n 2^-14 for both
  code classes); the min term is one more MMA pair with the min codes as A
  and the sub-block sums of x as B.
* block-diagonal engine for the 16-weight sub-block K-quants (Q2_K, Q6_K),
  read from their planar rows: a sub-block's 2-bit fields (Q2_K codes,
  Q6_K high parts) sit at bit kField[i] of one word, and W, W >> 2,
  rotr(W, 24), rotr(W, 24) >> 2 masked with 0x00300030 / 0x03000300 give
  positions (0,4)(1,5) | (2,6)(3,7) | (8,12)(9,13) | (10,14)(11,15) as fp16
  subnormals (Q6_K ORs in its low nibbles); lane t owns sub-block 4t + q of
  group q.
* ring engine (one or two vectors; also the MoE expert kernels): the 16 A
  rows are 8 weight rows x two halves of each code word (nibble positions
  0, 4, 2, 6 and 1, 5, 3, 7), lane (g, t) owns sub-blocks 2t, 2t+1 with the
  scale folded in by HMUL2; the 8 B columns are (half, vector, hi/lo), the
  x of a superblock scaled by 2^(15 - E) for |x| < 2^E; lanes t < 2 keep
  half 0 and t >= 2 half 1 of vector t & 1, and the min term is added per
  lane in float32 from the sub-block sums of x.
"""
import numpy as np
import pytest

import oracle
import synthetic

NIB_A, NIB_B = 0x000F000F, 0x00F000F0


def _h2(u):
    """uint32 -> the two fp16 halves (low, high) as float64, subnormals included."""
    return np.array([u & 0xFFFF, u >> 16], np.uint16).view(np.float16).astype(np.float64)


def _pack(a, b):
    """two floats -> uint32 of fp16 halves (round to nearest)."""
    h = np.array([a, b], np.float32).astype(np.float16).view(np.uint16)
    return int(h[0]) | (int(h[1]) << 16)


def _split(a, b):
    """fp32 pair -> (hi, lo) fp16 pairs: hi = fp16(v), lo = fp16(v - hi)."""
    a, b = np.float32(a), np.float32(b)
    ha, hb = np.float16(a), np.float16(b)
    return _pack(ha, hb), _pack(np.float32(a) - np.float32(ha), np.float32(b) - np.float32(hb))


def _hmul2(u, s):
    r = (_h2(u) * _h2(s)).astype(np.float16).view(np.uint16)
    return int(r[0]) | (int(r[1]) << 16)


def _mma(a_regs, b_regs):
    """C[16][8] = A[16][16] @ B[16][8] from per-lane registers."""
    A, B = np.zeros((16, 16)), np.zeros((16, 8))
    for lane in range(32):
        g, t = lane >> 2, lane & 3
        a0, a1, a2, a3 = a_regs[lane]
        A[g, 2 * t:2 * t + 2], A[g + 8, 2 * t:2 * t + 2] = _h2(a0), _h2(a1)
        A[g, 2 * t + 8:2 * t + 10], A[g + 8, 2 * t + 8:2 * t + 10] = _h2(a2), _h2(a3)
        b0, b1 = b_regs[lane]
        B[2 * t:2 * t + 2, g], B[2 * t + 8:2 * t + 10, g] = _h2(b0), _h2(b1)
    return A @ B


def _superblock_fields(packed_row, sb):
    """Q4_K superblock sb of a packed row: (d, dmin, scale codes, min codes,
    nibble word j of lane t -> words[t][j])."""
    b = packed_row[144 * sb:144 * (sb + 1)]
    d = float(np.frombuffer(bytes(b[0:2]), np.float16)[0])
    dmin = float(np.frombuffer(bytes(b[2:4]), np.float16)[0])
    stream = int.from_bytes(bytes(b[4:16]), "little")
    c = [(stream >> (6 * j)) & 63 for j in range(8)]
    m = [(stream >> (48 + 6 * j)) & 63 for j in range(8)]
    words = [[int.from_bytes(bytes(b[16 + 32 * t + 4 * j:20 + 32 * t + 4 * j]), "little") for j in range(8)]
             for t in range(4)]
    return d, dmin, c, m, words


def _exponent(xs):
    mx = float(np.max(np.abs(xs)))
    return int(np.floor(np.log2(mx))) if mx > 0 else 0


def _block_diagonal(packed, x, nsb):
    """One vector through the block-diagonal layout, 16 rows."""
    out = np.zeros(16)
    for sb in range(nsb):
        xs = x[256 * sb:256 * (sb + 1)].astype(np.float32)
        e = _exponent(xs)
        # B records: lane l stages positions 8l..8l+7 (sub-block s = l/4, word
        # i = l%4, owner o = s/2, group q = s%2) into MMA q*8 + 2i + mm
        rec = {}
        for l in range(32):
            s, i = l >> 2, l & 3
            q, o = s & 1, s >> 1
            v = xs[8 * l:8 * l + 8]
            hi, lo = [], []
            for k in range(4):
                f = np.float32(2.0 ** ((10 if k & 1 else 14) - e))
                h, w = _split(v[k] * f, v[k + 4] * f)
                hi.append(h)
                lo.append(w)
            for mm in range(2):
                rec[(q * 8 + 2 * i + mm, 2 * o)] = (hi[2 * mm], hi[2 * mm + 1])
                rec[(q * 8 + 2 * i + mm, 2 * o + 1)] = (lo[2 * mm], lo[2 * mm + 1])
        X = [float(np.sum(xs[32 * s:32 * s + 32], dtype=np.float32)) for s in range(8)]
        fields = [_superblock_fields(packed[r], sb) for r in range(16)]
        cs, ms = np.zeros(16), np.zeros(16)
        for q in range(2):
            C = np.zeros((16, 8))
            for mi in range(8):
                a_regs, b_regs = [], []
                for lane in range(32):
                    g, t = lane >> 2, lane & 3
                    wl, wh = fields[g][4][t][4 * q + mi // 2], fields[g + 8][4][t][4 * q + mi // 2]
                    if mi & 1:
                        wl, wh = wl >> 8, wh >> 8
                    a_regs.append((wl & NIB_A, wh & NIB_A, wl & NIB_B, wh & NIB_B))
                    col_owner = g >> 1
                    b_regs.append(rec[(q * 8 + mi, g)] if col_owner == t else (0, 0))
                C += _mma(a_regs, b_regs)
            for lane in range(32):
                g, t = lane >> 2, lane & 3
                for r in (g, g + 8):
                    _, _, c, m, _ = fields[r]
                    # lane (g, t) holds owner t's hi and lo columns of rows g, g + 8
                    cs[r] += c[2 * t + q] * (C[r, 2 * t] + C[r, 2 * t + 1])
                    ms[r] += m[2 * t + q] * X[2 * t + q]
        for r in range(16):
            d, dmin = fields[r][0], fields[r][1]
            out[r] += d * 2.0 ** (10 + e) * cs[r] - dmin * ms[r]
    return out


def _vector_column(packed, x, nsb):
    """8 vectors through the vector-column layout, 16 rows -> [16][8]."""
    nv = x.shape[0]
    out = np.zeros((16, 8))
    for sb in range(nsb):
        xs = x[:, 256 * sb:256 * (sb + 1)].astype(np.float32)
        main, minb, ps = {}, {}, np.zeros(8)
        for v in range(nv):
            e = _exponent(xs[v])
            f = np.float32(2.0 ** (14 - e))
            for l in range(32):
                tp, j = l >> 3, l & 7
                L = 4 * v + tp
                q = xs[v, 8 * l:8 * l + 8] * f
                h0, l0 = _split(q[0], q[4])
                h1, l1 = _split(q[1], q[5])
                h2, l2 = _split(q[2], q[6])
                h3, l3 = _split(q[3], q[7])
                main[(2 * j, L)] = ((h0, h1), (l0, l1))
                main[(2 * j + 1, L)] = ((h2, h3), (l2, l3))
            g9 = np.float32(2.0 ** (9 - e))
            for tp in range(4):
                X0 = np.float32(np.sum(xs[v, 64 * tp:64 * tp + 32], dtype=np.float32)) * g9
                X1 = np.float32(np.sum(xs[v, 64 * tp + 32:64 * tp + 64], dtype=np.float32)) * g9
                minb[4 * v + tp] = _split(X0, X1)
            ps[v] = 2.0 ** (e - 9)
        zero = ((0, 0), (0, 0))
        fields = [_superblock_fields(packed[r], sb) for r in range(16)]
        Cm = np.zeros((16, 8))
        for mi in range(16):
            j, h = mi // 2, mi % 2
            a_regs, bh, bl = [], [], []
            for lane in range(32):
                g, t = lane >> 2, lane & 3
                regs = []
                for r in (g, g + 8):
                    c = fields[r][2][2 * t + (j >= 4)]
                    w = fields[r][4][t][j] >> (8 * h)
                    regs.append((_hmul2(w & NIB_A, _pack(c * 1024.0, c * 1024.0)),
                                 _hmul2(w & NIB_B, _pack(c * 64.0, c * 64.0))))
                a_regs.append((regs[0][0], regs[1][0], regs[0][1], regs[1][1]))
                hi, lo = main.get((mi, lane), zero)
                bh.append(hi)
                bl.append(lo)
            Cm += _mma(a_regs, bh) + _mma(a_regs, bl)
        a_min = [(_pack(fields[lane >> 2][3][2 * (lane & 3)], fields[lane >> 2][3][2 * (lane & 3) + 1]),
                  _pack(fields[(lane >> 2) + 8][3][2 * (lane & 3)], fields[(lane >> 2) + 8][3][2 * (lane & 3) + 1]),
                  0, 0) for lane in range(32)]
        Cn = (_mma(a_min, [(minb.get(l, (0, 0))[0], 0) for l in range(32)])
              + _mma(a_min, [(minb.get(l, (0, 0))[1], 0) for l in range(32)]))
        for r in range(16):
            d, dmin = fields[r][0], fields[r][1]
            out[r] += ps * (512.0 * d * Cm[r] - dmin * Cn[r])
    return out[:, :nv]


KFIELD = [4, 8, 6, 10, 20, 24, 22, 26, 28, 0, 30, 2, 12, 16, 14, 18]
MASK_A, MASK_B = 0x00300030, 0x03000300
# x positions of MMA i in k-slots (2t, 2t+1) (class A) and (2t+8, 2t+9) (class B)
K16_POS = [(0, 4, 1, 5), (2, 6, 3, 7), (8, 12, 9, 13), (10, 14, 11, 15)]


def _rotr(w, s_):
    return ((w >> s_) | (w << (32 - s_))) & 0xFFFFFFFF


def _u32(b, off):
    return int.from_bytes(bytes(b[off:off + 4]), "little")


def _k16_subblock(fmt, row, nsb, sb, s_):
    """Planar row -> (code word W, nibble words (Q6_K) or None, scale code,
    min-term code, d, min-term factor) of sub-block s_ of superblock sb."""
    if fmt == oracle.Q2_K:
        W = _u32(row, 64 * sb + 4 * s_)
        sub = int(row[64 * nsb + 16 * sb + s_])
        fac = row[80 * nsb + 4 * sb:80 * nsb + 4 * sb + 4]
        d, dmin = (float(v) for v in np.frombuffer(bytes(fac), np.float16))
        return W, None, sub & 15, sub >> 4, d, dmin
    W = _u32(row, 128 * nsb + 64 * sb + 4 * s_)
    nib = (_u32(row, 128 * sb + 8 * s_), _u32(row, 128 * sb + 8 * s_ + 4))
    c = int(np.frombuffer(bytes(row[192 * nsb + 16 * sb + s_:192 * nsb + 16 * sb + s_ + 1]), np.int8)[0])
    d = float(np.frombuffer(bytes(row[208 * nsb + 2 * sb:208 * nsb + 2 * sb + 2]), np.float16)[0])
    # w = d c (u - 32): the offset term is 32 d times c sum(x)
    return W, nib, c, c, d, 32.0 * d


def _k16_pairs(fmt, W, nib, i):
    """Class-A and class-B fp16 pairs of MMA i from the masked words."""
    base = [W, W >> 2, _rotr(W, 24), _rotr(W, 24) >> 2][i]
    if fmt == oracle.Q2_K:
        return base & MASK_A, base & MASK_B
    n = [nib[0], nib[0] >> 8, nib[1], nib[1] >> 8][i]
    return (n & NIB_A) | (base & MASK_A), (n & NIB_B) | (base & MASK_B)


def _block_diagonal_k16(fmt, packed, x, nsb):
    """One vector of a Q2_K / Q6_K matrix through the block-diagonal layout,
    16 rows."""
    out = np.zeros(16)
    for sb in range(nsb):
        xs = x[256 * sb:256 * (sb + 1)].astype(np.float32)
        e = _exponent(xs)
        fA, fB = np.float32(2.0 ** (14 - e)), np.float32(2.0 ** (10 - e))
        ps = 2.0 ** ((6 if fmt == oracle.Q2_K else 10) + e)
        cs, ms = np.zeros(16), np.zeros(16)
        for q in range(4):
            fields = {(r, t): _k16_subblock(fmt, packed[r], nsb, sb, 4 * t + q) for r in range(16) for t in range(4)}
            C = np.zeros((16, 8))
            for i in range(4):
                pa0, pa1, pb0, pb1 = K16_POS[i]
                a_regs, b_regs = [], []
                for lane in range(32):
                    g, t = lane >> 2, lane & 3
                    lo, hi = _k16_pairs(fmt, *fields[(g, t)][:2], i), _k16_pairs(fmt, *fields[(g + 8, t)][:2], i)
                    a_regs.append((lo[0], hi[0], lo[1], hi[1]))
                    if (g >> 1) != t:  # column of another owner: the zero slot
                        b_regs.append((0, 0))
                        continue
                    v = xs[16 * (4 * t + q):16 * (4 * t + q) + 16]
                    part = g & 1
                    b_regs.append((_split(v[pa0] * fA, v[pa1] * fA)[part], _split(v[pb0] * fB, v[pb1] * fB)[part]))
                C += _mma(a_regs, b_regs)
            for lane in range(32):
                g, t = lane >> 2, lane & 3
                X = float(np.sum(xs[16 * (4 * t + q):16 * (4 * t + q) + 16], dtype=np.float32))
                for r in (g, g + 8):
                    _, _, c, k, _, _ = fields[(r, t)]
                    cs[r] += c * (C[r, 2 * t] + C[r, 2 * t + 1])
                    ms[r] += k * X
        for r in range(16):
            _, _, _, _, d, dmin = _k16_subblock(fmt, packed[r], nsb, sb, 0)
            out[r] += d * ps * cs[r] - dmin * ms[r]
    return out


def _bound_exponent(amax):
    """E with |x| < 2^E from the float32 exponent field (zero reads as the
    smallest normal binade)."""
    eb = int(np.array([amax], np.float32).view(np.uint32)[0] >> 23) & 0xFF
    return max(eb, 1) - 126


def _ring(packed, x, nsb):
    """One or two vectors through the ring engine's layout, 8 rows -> [8][nv]."""
    nv = x.shape[0]
    out = np.zeros((8, nv))
    for sb in range(nsb):
        xs = x[:, 256 * sb:256 * (sb + 1)].astype(np.float32)
        q, fs, X = [], [], []
        for v in range(nv):
            sig = min(126, max(-112, 15 - _bound_exponent(float(np.max(np.abs(xs[v]))))))
            q.append(xs[v] * np.float32(2.0 ** sig))
            fs.append(2.0 ** (14 - sig))
            X.append([float(np.sum(xs[v, 32 * s_:32 * s_ + 32], dtype=np.float32)) for s_ in range(8)])
        fields = [_superblock_fields(packed[r], sb) for r in range(8)]
        C = np.zeros((16, 8))
        for j in range(8):
            a_regs, b_regs = [], []
            for lane in range(32):
                g, t = lane >> 2, lane & 3
                _, _, c, _, words = fields[g]
                code = c[2 * t + (j >> 2)]
                mlo, mhi = _pack(code * 1024.0, code * 1024.0), _pack(code * 64.0, code * 64.0)
                w = words[t][j]
                a_regs.append((_hmul2(w & NIB_A, mlo), _hmul2(w & NIB_B, mhi),
                               _hmul2((w >> 8) & NIB_A, mlo), _hmul2((w >> 8) & NIB_B, mhi)))
                # B column g = (half h, vector v, lo): x of sub-block 2t + j/4,
                # word j % 4, at the positions of half h
                h, v, lo = g >> 2, (g >> 1) & 1, g & 1
                if v >= nv:
                    b_regs.append((0, 0))
                    continue
                base = 32 * (2 * t + (j >> 2)) + 8 * (j & 3)
                qv = q[v][base:base + 8]
                b_regs.append((_split(qv[h], qv[h + 4])[lo], _split(qv[h + 2], qv[h + 6])[lo]))
            C += _mma(a_regs, b_regs)
        for lane in range(32):
            g, t = lane >> 2, lane & 3
            d, dmin, _, m, _ = fields[g]
            cv = t & 1
            s_ = C[g, 2 * t] + C[g, 2 * t + 1] if t < 2 else C[g + 8, 2 * t] + C[g + 8, 2 * t + 1]
            if cv < nv:
                out[g, cv] += d * s_ * fs[cv]
            for v in range(nv):
                out[g, v] -= dmin * (m[2 * t] * X[v][2 * t] + m[2 * t + 1] * X[v][2 * t + 1])
    return out


def _case(seed, nsb, nv, spread):
    W = synthetic.student_t((16, 256 * nsb), seed=seed).numpy()
    packed = oracle.quantize(oracle.Q4_K, W)
    x = synthetic.normal((nv, 256 * nsb), seed=seed + 1).numpy()
    x = (x * np.float32(10.0) ** np.linspace(-spread, spread, nv, dtype=np.float32)[:, None]).astype(np.float32)
    return packed, x


def _assert_close(got, packed, x, cols, fmt=oracle.Q4_K):
    ref = oracle.gemv_f64(fmt, packed, x, cols)       # [nv][rows]
    bound = oracle.gemv_bound(fmt, packed, x, cols)
    err = np.abs(got - ref)
    assert (err <= 1e-6 * bound + 1e-30).all(), (err / (bound + 1e-30)).max()


def test_block_diagonal_layout_matches_oracle():
    for seed, nsb in ((3, 1), (5, 2)):
        packed, x = _case(seed, nsb, 1, 0.0)
        got = _block_diagonal(packed, x[0], nsb)
        _assert_close(got[None, :], packed, x, 256 * nsb)


def test_vector_column_layout_matches_oracle():
    for seed, nsb, nv, spread in ((7, 1, 8, 3.0), (9, 2, 5, 1.0), (11, 1, 2, 0.0)):
        packed, x = _case(seed, nsb, nv, spread)
        got = _vector_column(packed, x, nsb)
        _assert_close(got.T, packed, x, 256 * nsb)


@pytest.mark.parametrize("fmt", [oracle.Q2_K, oracle.Q6_K])
def test_block_diagonal_k16_layout_matches_oracle(fmt):
    for seed, nsb in ((23, 1), (25, 3)):
        W = synthetic.student_t((16, 256 * nsb), seed=seed).numpy()
        packed = oracle.quantize(fmt, W)
        x = synthetic.normal((1, 256 * nsb), seed=seed + 1).numpy()
        got = _block_diagonal_k16(fmt, packed, x[0], nsb)
        _assert_close(got[None, :], packed, x, 256 * nsb, fmt)


def test_k16_field_table_gives_the_mma_positions():
    """W, W >> 2, rotr(W, 24) and rotr(W, 24) >> 2 bring exactly the fields
    of MMA i's positions (kField of K16_POS[i]) to the mask bits: bit 4 / 20
    (class A, low / high fp16 half) and 8 / 24 (class B)."""
    forms = [lambda w: w, lambda w: w >> 2, lambda w: _rotr(w, 24), lambda w: _rotr(w, 24) >> 2]
    for i, f in enumerate(forms):
        for slot, target in enumerate((4, 20, 8, 24)):
            src = [b for b in range(32) if f(1 << b) & (1 << target)]
            assert src == [KFIELD[K16_POS[i][slot]]], (i, slot, src)
    assert sorted(KFIELD) == list(range(0, 32, 2))   # 16 disjoint 2-bit fields


def test_block_diagonal_k16_model_catches_moved_fields():
    """The model reads field positions from the bits: exchanging the codes
    of positions 8 and 9 (bits 28 and 0) in every word breaks the match."""
    W = synthetic.student_t((16, 256), seed=27).numpy()
    packed = oracle.quantize(oracle.Q2_K, W)
    x = synthetic.normal((1, 256), seed=28).numpy()
    ref = oracle.gemv_f64(oracle.Q2_K, packed, x, 256)
    bound = oracle.gemv_bound(oracle.Q2_K, packed, x, 256)
    bad_packed = packed.copy()
    for r in range(16):
        for s_ in range(16):
            w = _u32(bad_packed[r], 4 * s_)
            a, b = (w >> 28) & 3, w & 3
            w = (w & ~((3 << 28) | 3) & 0xFFFFFFFF) | (b << 28) | a
            bad_packed[r, 4 * s_:4 * s_ + 4] = np.frombuffer(w.to_bytes(4, "little"), np.uint8)
    bad = _block_diagonal_k16(oracle.Q2_K, bad_packed, x[0], 1)
    assert (np.abs(bad[None, :] - ref) > 1e-3 * bound).any()


def test_ring_layout_matches_oracle():
    for seed, nsb, nv, spread in ((15, 1, 1, 0.0), (17, 2, 2, 3.0), (19, 3, 2, 0.0)):
        packed, x = _case(seed, nsb, nv, spread)
        packed = packed[:8]
        got = _ring(packed, x, nsb)
        _assert_close(got.T, packed, x, 256 * nsb)


def test_ring_layout_model_catches_a_wrong_nibble_mask():
    """The odd nibble positions (A registers 1 and 3) read through the even
    positions' mask, a plausible slip, breaks the match by far more than
    the bound."""
    packed, x = _case(21, 1, 2, 0.0)
    packed = packed[:8]
    ref = oracle.gemv_f64(oracle.Q4_K, packed, x, 256)
    bound = oracle.gemv_bound(oracle.Q4_K, packed, x, 256)
    global NIB_B
    saved = NIB_B
    try:
        NIB_B = NIB_A  # odd nibble positions read the even ones
        bad = _ring(packed, x, 1).T
    finally:
        NIB_B = saved
    assert (np.abs(bad - ref) > 1e-3 * bound).any()


def test_layout_models_catch_a_wrong_slot():
    """The models are not vacuous: moving the class-B scale of the
    vector-column layout from c 2^6 to c 2^10 (a plausible slip) or
    dropping the min term breaks the match by far more than the bound."""
    packed, x = _case(13, 1, 3, 0.0)
    ref = oracle.gemv_f64(oracle.Q4_K, packed, x, 256)
    bound = oracle.gemv_bound(oracle.Q4_K, packed, x, 256)
    global NIB_B
    saved = NIB_B
    try:
        NIB_B = NIB_A  # the class-B slots now read class-A nibbles
        bad = _vector_column(packed, x, 1).T
    finally:
        NIB_B = saved
    assert (np.abs(bad - ref) > 1e-3 * bound).any()
