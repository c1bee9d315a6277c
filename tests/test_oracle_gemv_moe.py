"""Pins for the GEMV and MoE oracles: brute force on tiny shapes, closed
forms, invariants and special cases."""
import math

import numpy as np
import pytest

import oracle
from oracle import Q8_0, Q4_0, Q4_1, Q4_K
from oracle.moe import MoEWeights


def _rand_w(rng, rows, cols):
    return (rng.standard_t(5, (rows, cols)) * 0.02).astype(np.float32)


# ------------------------------------------------------------------ GEMV
@pytest.mark.parametrize("fmt", oracle.FORMATS)
def test_gemv_brute_force(fmt):
    """Python loops in float64 over the dequantized matrix, 3 rows x 256 cols x 2 vectors."""
    rng = np.random.default_rng(fmt)
    W = _rand_w(rng, 3, 256)
    x = rng.standard_normal((2, 256)).astype(np.float32)
    p = oracle.quantize(fmt, W)
    deq = oracle.dequantize(fmt, p, 256)
    y = oracle.gemv_f64(fmt, p, x, 256)
    A = oracle.gemv_bound(fmt, p, x, 256)
    assert y.shape == (2, 3)
    for v in range(2):
        for i in range(3):
            s = 0.0
            a = 0.0
            for j in range(256):
                t = float(deq[i, j]) * float(x[v, j])
                s += t
                a += abs(t)
            assert y[v, i] == pytest.approx(s, rel=1e-12, abs=1e-15)
            assert A[v, i] == pytest.approx(a, rel=1e-12)


@pytest.mark.parametrize("fmt", oracle.FORMATS)
def test_gemv_against_exact_rational_sum(fmt):
    """Both float64 GEMV oracles (numpy and C++) against the exact sum in
    rational arithmetic: the dequantized float32 weights and a dyadic x are
    exact as fractions, so the float64 results may differ from the exact
    value only by float64 summation error (n * 2^-53 of sum |w x|)."""
    from fractions import Fraction

    from oracle import cref
    rng = np.random.default_rng(40 + fmt)
    cols = 512
    W = _rand_w(rng, 3, cols)
    x = (rng.integers(-64, 65, (2, cols)) * 2.0 ** -5).astype(np.float32)
    p = oracle.quantize(fmt, W)
    deq = oracle.dequantize(fmt, p, cols)
    y_np = oracle.gemv_f64(fmt, p, x, cols)
    y_c, _ = cref.gemv_f64(fmt, p, x, cols)
    for v in range(2):
        for i in range(3):
            terms = [Fraction(float(deq[i, j])) * Fraction(float(x[v, j])) for j in range(cols)]
            exact = sum(terms, Fraction(0))
            A = float(sum(abs(t) for t in terms))
            tol = cols * 2.0 ** -53 * A
            assert abs(Fraction(float(y_np[v, i])) - exact) <= Fraction(tol), (fmt, v, i)
            assert abs(Fraction(float(y_c[v, i])) - exact) <= Fraction(tol), (fmt, v, i)


def test_gemv_one_hot_gives_column():
    rng = np.random.default_rng(1)
    W = _rand_w(rng, 5, 512)
    for fmt in oracle.FORMATS:
        p = oracle.quantize(fmt, W)
        deq = oracle.dequantize(fmt, p, 512)
        for j in (0, 31, 32, 255, 256, 511):
            x = np.zeros(512, np.float32)
            x[j] = 1.0
            assert np.array_equal(oracle.gemv_f64(fmt, p, x, 512)[0], deq[:, j].astype(np.float64))


def test_gemv_linearity_and_quantized_is_close_to_dense():
    rng = np.random.default_rng(2)
    W = _rand_w(rng, 64, 1024)
    x1 = rng.standard_normal(1024).astype(np.float32)
    x2 = rng.standard_normal(1024).astype(np.float32)
    for fmt in oracle.FORMATS:
        p = oracle.quantize(fmt, W)
        y = oracle.gemv_f64(fmt, p, np.stack([x1, x2, x1 + x2]), 1024)
        A = oracle.gemv_bound(fmt, p, np.stack([x1, x2]), 1024)
        # x1 + x2 is rounded to float32 once: 2^-24 relative per term
        assert (np.abs(y[0] + y[1] - y[2]) <= 2.0 ** -23 * (A[0] + A[1])).all()
        dense = W.astype(np.float64) @ x1.astype(np.float64)
        rel = np.linalg.norm(y[0] - dense) / np.linalg.norm(dense)
        # the output error follows the weight error (page: 0.0068 .. 0.108;
        # 2-bit codes: about 0.36)
        assert rel < {Q8_0: 0.02, oracle.Q2_K: 0.45}.get(fmt, 0.25)


# ------------------------------------------------------------------ router / top-K
def test_topk_against_rank_counting():
    """Selected set = experts beaten by fewer than K others (ties -> lower index)."""
    rng = np.random.default_rng(4)
    for trial in range(20):
        E = 12
        l = np.round(rng.standard_normal((3, E)), 1)   # rounding creates ties
        for K in (1, 3, 8, 12):
            idx = oracle.topk_select(l, K)
            for t in range(3):
                rank = [sum(1 for f in range(E) if l[t, f] > l[t, e] or (l[t, f] == l[t, e] and f < e))
                        for e in range(E)]
                want = sorted(range(E), key=lambda e: rank[e])[:K]
                assert idx[t].tolist() == want


def test_softmax_and_combine_weights():
    rng = np.random.default_rng(6)
    l = rng.standard_normal((4, 16)) * 3
    p = oracle.softmax_f64(l)
    assert np.allclose(p.sum(1), 1.0, atol=1e-15)
    # closed form on a two-expert case: softmax(a, b)_0 = 1 / (1 + e^(b - a))
    q = oracle.softmax_f64(np.array([[1.0, 2.5]]))
    assert q[0, 0] == pytest.approx(1 / (1 + math.exp(1.5)), rel=1e-14)
    idx = oracle.topk_select(l, 16)
    w = oracle.combine_weights(l, idx, True)
    assert np.allclose(w.sum(1), 1)
    assert np.allclose(np.sort(w, 1), np.sort(p, 1))        # K = E keeps every expert
    w4 = oracle.combine_weights(l, oracle.topk_select(l, 4), False)
    assert np.allclose(w4, np.sort(p, 1)[:, ::-1][:, :4])


def test_router_logits_closed_form():
    """R is a non-square shifted identity (row e picks column e + 1), so the
    logits are x[e + 1] + bias[e]: a transposed R, a dropped or negated bias
    or a wrong shift gives other numbers."""
    E, H = 3, 5
    R = np.zeros((E, H), np.float32)
    for e in range(E):
        R[e, e + 1] = 1.0
    x = np.array([[1.0, 2.0, 3.0, 4.0, 5.0], [-1.0, 0.5, -0.25, 8.0, 0.0]], np.float32)
    bias = np.array([10.0, -1.0, 0.5], np.float32)
    assert oracle.router_logits_f64(R, x).tolist() == [[2.0, 3.0, 4.0], [0.5, -0.25, 8.0]]
    assert oracle.router_logits_f64(R, x, bias).tolist() == [[12.0, 2.0, 4.5], [10.5, -1.25, 8.5]]


def test_rmsnorm_closed_form():
    x = np.array([[3.0, 4.0]])
    # mean of squares 12.5
    assert np.allclose(oracle.rmsnorm_f64(x, 0.0), x / math.sqrt(12.5))


# ------------------------------------------------------------------ expert / MoE
def _identity_expert(H, scale_gate, scale_up, scale_down, shift):
    """Q8_0 expert whose dequantized matrices are scaled identities and a
    cyclic shift (values 127 * 2^-e are exact in Q8_0)."""
    G = np.eye(H, dtype=np.float32) * scale_gate
    U = np.eye(H, dtype=np.float32) * scale_up
    D = np.roll(np.eye(H, dtype=np.float32), shift, axis=1) * scale_down   # D[i, (i+shift)%H]
    gu = oracle.quantize(Q8_0, np.concatenate([G, U]))
    d = oracle.quantize(Q8_0, D)
    return gu, d


def test_expert_closed_form():
    """down(silu(gate x) * up x) with gate = c I, up = 2c I, down = c P (shift by 1)."""
    H = 32
    c = 127 / 128
    gu, d = _identity_expert(H, c, 2 * c, c, 1)
    x = np.linspace(-3, 3, H).astype(np.float32)
    o, g, u, h = oracle.expert_forward_f64(Q8_0, gu, d, H, H, x)
    silu = lambda v: v / (1 + np.exp(-v))
    hh = silu(c * x.astype(np.float64)) * (2 * c * x.astype(np.float64))
    assert np.allclose(g[0], c * x)
    assert np.allclose(u[0], 2 * c * x)
    assert np.allclose(h[0], hh, rtol=1e-14)
    assert np.allclose(o[0], c * np.roll(hh, -1), rtol=1e-14)     # o_i = c * h_{i+1}


def _random_moe(rng, fmt, E, H, I, shared=True, gate_vec=False, bias=False, norm=True):
    R = (rng.standard_t(5, (E, H)) * 0.02).astype(np.float32)
    gu = np.stack([oracle.quantize(fmt, _rand_w(rng, 2 * I, H)) for _ in range(E)])
    dn = np.stack([oracle.quantize(fmt, _rand_w(rng, H, I)) for _ in range(E)])
    mw = MoEWeights(fmt=fmt, hidden=H, inter=I, router=R, gate_up=gu, down=dn, norm_topk=norm)
    if bias:
        mw.router_bias = rng.standard_normal(E).astype(np.float32)
    if shared:
        mw.shared_gate_up = oracle.quantize(fmt, _rand_w(rng, 2 * I, H))
        mw.shared_down = oracle.quantize(fmt, _rand_w(rng, H, I))
        if gate_vec:
            mw.shared_gate_vec = (rng.standard_normal(H) * 0.05).astype(np.float32)
    return mw


def test_moe_zero_experts_is_identity():
    rng = np.random.default_rng(8)
    mw = _random_moe(rng, Q4_K, 8, 256, 256)
    mw.gate_up = np.stack([oracle.quantize(Q4_K, np.zeros((512, 256), np.float32))] * 8)
    mw.down = np.stack([oracle.quantize(Q4_K, np.zeros((256, 256), np.float32))] * 8)
    mw.shared_down = oracle.quantize(Q4_K, np.zeros((256, 256), np.float32))
    x = rng.standard_normal((3, 256)).astype(np.float32)
    r = oracle.moe_forward_f64(mw, x, 2)
    assert np.array_equal(r.y, x.astype(np.float64))


def test_moe_matches_per_expert_sum():
    """y = x + sum_k w_k expert_k(x) + sigmoid(g.x) shared(x), assembled by hand."""
    rng = np.random.default_rng(10)
    for norm in (True, False):
        mw = _random_moe(rng, Q4_K, 6, 256, 256, gate_vec=True, bias=True, norm=norm)
        x = rng.standard_normal((2, 256)).astype(np.float32)
        r = oracle.moe_forward_f64(mw, x, 3)
        for t in range(2):
            l = x[t].astype(np.float64) @ mw.router.astype(np.float64).T + mw.router_bias
            order = np.argsort(-l, kind="stable")[:3]
            assert r.idx[t].tolist() == order.tolist()
            p = np.exp(l - l.max())
            p /= p.sum()
            w = p[order] / (p[order].sum() if norm else 1.0)
            y = x[t].astype(np.float64).copy()
            for k, e in enumerate(order):
                y += w[k] * oracle.expert_forward_f64(Q4_K, mw.gate_up[e], mw.down[e], 256, 256, x[t])[0][0]
            gs = 1 / (1 + math.exp(-(x[t].astype(np.float64) @ mw.shared_gate_vec)))
            y += gs * oracle.expert_forward_f64(Q4_K, mw.shared_gate_up, mw.shared_down, 256, 256, x[t])[0][0]
            assert np.allclose(r.y[t], y, rtol=1e-12, atol=1e-12)


def test_moe_prenorm_reads_normalized_input():
    rng = np.random.default_rng(12)
    mw = _random_moe(rng, Q4_0, 4, 256, 256)
    x = (rng.standard_normal((2, 256)) * 7).astype(np.float32)
    r = oracle.moe_forward_f64(mw, x, 2, rms_eps=1e-6)
    xn = x / np.sqrt((x.astype(np.float64) ** 2).mean(1, keepdims=True) + np.float32(1e-6))
    assert np.allclose(r.xin, xn, rtol=1e-14)
    assert np.allclose(np.sqrt((r.xin ** 2).mean(1)), 1.0, rtol=1e-6)
    r2 = oracle.moe_forward_f64(mw, xn, 2)          # xn is rounded to float32 here
    assert (r.idx == r2.idx).all()
    # experts see the normalized input, the residual stays x
    assert np.allclose(r.y - x, r2.y - xn.astype(np.float32), rtol=1e-5, atol=1e-7)


def test_moe_single_expert_all_tokens():
    """K = 1 over one expert: every token goes to expert 0 with weight 1."""
    rng = np.random.default_rng(13)
    mw = _random_moe(rng, Q4_1, 1, 256, 256, shared=False)
    x = rng.standard_normal((4, 256)).astype(np.float32)
    r = oracle.moe_forward_f64(mw, x, 1)
    assert (r.idx == 0).all() and np.allclose(r.w, 1.0)
    o = oracle.expert_forward_f64(Q4_1, mw.gate_up[0], mw.down[0], 256, 256, x)[0]
    assert np.allclose(r.y, x + o, rtol=1e-12)


def _diag_q8(value: float, n: int) -> np.ndarray:
    """Q8_0 packing of value * identity (n x n): each row's only nonzero
    block holds `value` at the diagonal; value = 127 * 2^-p packs exactly
    (scale 2^-p, code 127)."""
    W = np.zeros((n, n), np.float32)
    np.fill_diagonal(W, value)
    return oracle.quantize(oracle.Q8_0, W)


def test_moe_combine_and_sigmoid_gate_closed_form():
    """Pins the weighted combine and the sigmoid shared gate with values
    worked out by hand, independent of the oracle's own expert code.

    Two routed experts with diagonal gate, up and down matrices (every
    entry exactly representable) and one shared expert.  Expert e maps
    x_j to o_j = c_e * (a_e x_j) / (1 + exp(-a_e x_j)) * (b_e x_j).  The
    router sends x_0 = 1 to logits (ln 3, 0), so the softmax weights are
    exactly (3/4, 1/4); with both chosen and renormalised they stay
    (3/4, 1/4), with one chosen and renormalised it is 1, without
    renormalisation 3/4.  The shared gate vector is orthogonal to x, so
    sigmoid(g . x) = 1/2."""
    n = 32
    vals = {0: (127 * 2.0 ** -7, 127 * 2.0 ** -8, 127 * 2.0 ** -6),     # a, b, c per expert
            1: (127 * 2.0 ** -6, 127 * 2.0 ** -7, 127 * 2.0 ** -9),
            "s": (127 * 2.0 ** -8, 127 * 2.0 ** -6, 127 * 2.0 ** -7)}
    gu = {k: np.concatenate([_diag_q8(a, n), _diag_q8(b, n)]) for k, (a, b, _) in vals.items()}
    dn = {k: _diag_q8(c, n) for k, (_, _, c) in vals.items()}
    x = np.linspace(-1.5, 1.25, n).astype(np.float32)
    x[0] = 1.0
    x[1] = x[2] = np.float32(0.5)
    R = np.zeros((2, n), np.float32)
    R[0, 0] = np.float32(np.log(3.0))          # logit of expert 0: ln 3 * x_0
    g = np.zeros(n, np.float32)
    g[1], g[2] = 1.0, -1.0                      # g . x = x_1 - x_2 = 0
    lnw = float(np.float32(np.log(3.0)))        # the logit as stored (float32)
    p0 = np.exp(lnw) / (np.exp(lnw) + 1.0)      # 3/4 up to float32(ln 3)

    def expert(k):
        a, b, c = vals[k]
        xd = x.astype(np.float64)
        return c * (a * xd) / (1.0 + np.exp(-a * xd)) * (b * xd)

    mw = MoEWeights(fmt=oracle.Q8_0, hidden=n, inter=n, router=R,
                    gate_up=np.stack([gu[0], gu[1]]), down=np.stack([dn[0], dn[1]]),
                    shared_gate_up=gu["s"], shared_down=dn["s"], shared_gate_vec=g)
    for topk, norm, w in ((2, True, (p0, 1 - p0)), (1, True, (1.0,)), (1, False, (p0,))):
        mw.norm_topk = norm
        r = oracle.moe_forward_f64(mw, x[None], topk)
        assert r.idx[0].tolist() == [0, 1][:topk]
        assert np.allclose(r.w[0], w, rtol=1e-15, atol=0)
        assert r.shared_gate[0] == 0.5
        y = x.astype(np.float64) + sum(wk * expert(k) for k, wk in enumerate(w)) + 0.5 * expert("s")
        assert np.allclose(r.y[0], y, rtol=1e-13, atol=1e-15)
    assert abs(p0 - 0.75) < 1e-7
    # a router bias of (0, ln 9) lifts expert 1 over expert 0: logits
    # (ln 3, ln 9), order [1, 0], weights 9/12 and 3/12
    mw.router_bias = np.array([0.0, np.log(9.0)], np.float32)
    mw.norm_topk = True
    lb = float(np.float32(np.log(9.0)))
    q1 = np.exp(lb) / (np.exp(lb) + np.exp(lnw))
    r = oracle.moe_forward_f64(mw, x[None], 2)
    assert r.idx[0].tolist() == [1, 0]
    assert np.allclose(r.w[0], (q1, 1 - q1), rtol=1e-15, atol=0)
    assert abs(q1 - 0.75) < 1e-7
    y = x.astype(np.float64) + q1 * expert(1) + (1 - q1) * expert(0) + 0.5 * expert("s")
    assert np.allclose(r.y[0], y, rtol=1e-13, atol=1e-15)
