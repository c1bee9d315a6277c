"""Pins for the plain C++ oracle (oracle/epq_ref.cpp) against what the pages
and the mathematics fix, and its agreement with the numpy oracle.

* fp16 encoding: all 2^32 float32 bit patterns against torch's IEEE
  round-to-nearest-even conversion (NaN compared as NaN);
* the handbook's printed table ("GGUF 的量化格式"): relative errors on the
  page's own sample, to 4 decimals;
* the hand-worked blocks of tests/golden/hand_blocks.txt, byte for byte;
* codes are the exhaustive-search nearest grid points;
* the numpy oracle (written separately, vectorised) gives the same bytes and
  the same dequantized bits on random and degenerate blocks;
* the float64 GEMV equals a brute-force float64 sum; the float32 GEMV (the
  CPU baseline) is within 1e-5 of sum |w x| and does not depend on the
  thread count.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import Q8_0, Q4_0, Q4_1, Q4_K, cref

from test_oracle_formats import _brute_codes, _hex

NAME = {"Q8_0": Q8_0, "Q4_0": Q4_0, "Q4_1": Q4_1, "Q4_K": Q4_K}


def test_fp16_encoding_all_float32_inputs():
    chunk = 1 << 27
    torch.set_num_threads(max(1, min(16, torch.get_num_threads())))
    for first in range(0, 1 << 32, chunk):
        bits = torch.arange(first, first + chunk, dtype=torch.int64).to(torch.int32)
        f = bits.view(torch.float32)
        ref = f.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
        ours = cref.f16_of_bits(first, chunk)
        bad = ours != ref
        if bad.any():
            # NaN encodings may differ in payload: both must be NaN
            ref_nan = (ref[bad] & 0x7C00) == 0x7C00
            ours_nan = (ours[bad] & 0x7C00) == 0x7C00
            assert (ref[bad] & 0x3FF).all() and (ours[bad] & 0x3FF).all() and ref_nan.all() and ours_nan.all(), \
                hex(first + int(np.flatnonzero(bad)[0]))


def test_fp16_decoding_all_halves():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    ours = np.array([cref.lib().eref_f16_to_f32(int(v)) for v in h], np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(ref[finite].view(np.uint32), ours[finite].view(np.uint32))
    assert np.array_equal(np.isnan(ref), np.isnan(ours))


def test_page2_relative_errors(golden):
    _, rows = golden("page2_formats.txt")
    w = synthetic.page2_sample().numpy().astype(np.float32)
    for name, bpw, rel in rows:
        fmt = NAME[name]
        packed = cref.quantize(fmt, w.reshape(4096, 256), threads=4)
        assert 8 * packed.size / w.size == pytest.approx(float(bpw), abs=1e-12)
        deq = cref.dequantize(fmt, packed, 256).reshape(-1).astype(np.float64)
        err = np.linalg.norm(deq - w) / np.linalg.norm(w.astype(np.float64))
        assert f"{err:.4f}" == rel, (name, err)


def test_hand_blocks(golden):
    g, _ = golden("hand_blocks.txt")
    c = [int(v) for v in g["q4k_values_c"]]
    k = [int(v) for v in g["q4k_values_k"]]
    n = list(range(16)) + list(range(15, -1, -1))
    x = np.array([[nn * (c[s] / 64) - k[s] / 128 for s in range(8) for nn in n]], np.float32)
    blk = cref.quantize(Q4_K, x)[0].tobytes()
    assert blk[0:2] == _hex(g["q4k_d"]) and blk[2:4] == _hex(g["q4k_dmin"])
    assert blk[4:16] == _hex(g["q4k_scales"])
    for s in range(8):
        assert blk[16 + 16 * s:32 + 16 * s] == _hex(g["q4k_qs"]), s
    assert np.array_equal(cref.dequantize(Q4_K, np.frombuffer(blk, np.uint8)[None], 256), x)

    q = [-127, -64, -1, 0] + list(range(1, 29))
    blk = cref.quantize(Q8_0, np.array([q], np.float32) / 16)[0].tobytes()
    assert blk[0:2] == _hex(g["q8_d"]) and blk[2:34] == _hex(g["q8_q"])

    base = np.array([((j % 16) - 8) / 4 for j in range(32)], np.float32)
    a = base.copy()
    a[5] = 2.0
    blk = cref.quantize(Q4_0, a[None])[0].tobytes()
    assert blk[0:2] == _hex(g["q40a_d"]) and blk[2:] == _hex(g["q40a_qs"])
    b = base.copy()
    b[0], b[5] = 2.0, -2.0
    blk = cref.quantize(Q4_0, b[None])[0].tobytes()
    assert blk[0:2] == _hex(g["q40b_d"]) and blk[2:] == _hex(g["q40b_qs"])

    x = np.array([[-1 + (j % 16) / 4 for j in range(32)]], np.float32)
    blk = cref.quantize(Q4_1, x)[0].tobytes()
    assert blk[0:2] == _hex(g["q41_d"]) and blk[2:4] == _hex(g["q41_m"]) and blk[4:20] == _hex(g["q41_qs"])


def test_codes_are_nearest_grid_points():
    rng = np.random.default_rng(17)
    x = (rng.standard_t(5, (4, 256)) * 0.02).astype(np.float32)
    F = oracle.formats._F
    p = cref.quantize(Q4_1, x).reshape(-1, 20)
    for b in range(0, p.shape[0], 3):
        d, m = F(p[b, 0:2].view("<f2"))[0], F(p[b, 2:4].view("<f2"))[0]
        n = oracle.formats._unpack_nibbles(p[b:b + 1, 4:])[0].astype(int)
        assert n.tolist() == _brute_codes(x.reshape(-1, 32)[b], d, m, 0, 15)
    p = cref.quantize(Q4_K, x).reshape(-1, 144)
    for b in range(p.shape[0]):
        d, dmin = F(p[b, 0:2].view("<f2"))[0], F(p[b, 2:4].view("<f2"))[0]
        c, k = oracle.formats._unpack_scales(p[b:b + 1, 4:16])
        xs = x.reshape(-1, 8, 32)[b]
        for s in range(8):
            S = np.float32(d * np.float32(c[0, s]))
            M = np.float32(dmin * np.float32(k[0, s]))
            n = oracle.formats._unpack_nibbles(p[b:b + 1, 16 + 16 * s:32 + 16 * s])[0].astype(int)
            assert n.tolist() == _brute_codes(xs[s], S, -M, 0, 15), (b, s)


def _degenerate(rows, cols, seed):
    W = synthetic.student_t((rows, cols), seed=seed).numpy()
    W[0, :64] = 0.0
    W[1, :64] = -0.0
    W[2, :cols] = 0.5
    W[3, :cols] = -0.25
    W[4, :cols] = np.abs(W[4, :cols])
    W[5, 0:32] = np.float32(2.0 ** -24)        # fp16-subnormal factors
    W[5, 32:64] = np.float32(-3 * 2.0 ** -20)
    W[6, :32] = np.where(np.arange(32) % 2 == 0, 1.0, -1.0)   # Q4_0 sign tie
    return W


@pytest.mark.parametrize("fmt", oracle.FORMATS)
@pytest.mark.parametrize("rows,cols", [(8, 256), (19, 512), (40, 4096)])
def test_numpy_and_cpp_oracles_agree(fmt, rows, cols):
    W = _degenerate(rows, cols, seed=rows * 31 + cols + fmt)
    a = oracle.quantize(fmt, W)
    b = cref.quantize(fmt, W, threads=3)
    assert np.array_equal(a, b)
    da = oracle.dequantize(fmt, a, cols)
    db = cref.dequantize(fmt, b, cols)
    assert np.array_equal(da.view(np.uint32), db.view(np.uint32))


@pytest.mark.parametrize("fmt", oracle.FORMATS)
def test_gemv_f64_brute_force(fmt):
    rows, cols = 5, 512
    W = synthetic.student_t((rows, cols), seed=70 + fmt).numpy()
    x = synthetic.normal((2, cols), seed=71).numpy()
    p = cref.quantize(fmt, W)
    deq = cref.dequantize(fmt, p, cols).astype(np.float64)
    y, A = cref.gemv_f64(fmt, p, x, cols, threads=2)
    for v in range(2):
        for i in range(rows):
            ref = 0.0
            mag = 0.0
            for j in range(cols):
                t = deq[i, j] * float(x[v, j])
                ref += t
                mag += abs(t)
            assert y[v, i] == ref and A[v, i] == mag
    # a one-hot x returns one dequantized column, exactly
    e = np.zeros((1, cols), np.float32)
    e[0, 37] = 1.0
    assert np.array_equal(cref.gemv_f64(fmt, p, e, cols)[0][0], deq[:, 37])


@pytest.mark.parametrize("fmt", oracle.FORMATS)
def test_gemv_f32_within_bound_and_thread_invariant(fmt):
    rows, cols = 300, 1024
    W = synthetic.student_t((rows, cols), seed=80 + fmt).numpy()
    x = synthetic.normal((3, cols), seed=81).numpy()
    p = cref.quantize(fmt, W, threads=4)
    y64, A = cref.gemv_f64(fmt, p, x, cols, threads=4)
    ys = [cref.gemv_f32(fmt, p, x, cols, threads=t) for t in (1, 2, 7)]
    for y in ys:
        assert np.array_equal(y, ys[0])
    assert (np.abs(ys[0] - y64) <= 1e-5 * A).all()


def test_quantize_thread_invariant():
    W = synthetic.student_t((97, 2048), seed=90).numpy()
    for fmt in oracle.FORMATS:
        assert np.array_equal(cref.quantize(fmt, W, threads=1), cref.quantize(fmt, W, threads=5))
