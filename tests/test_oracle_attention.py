"""Pins for the decode-attention oracle against closed forms: one position
returns its value row; two scores ln 3 apart give weights 3/4 and 1/4;
equal scores give the mean of the values; a position 10 below the maximum
(below ln(1e-4) = -9.21) is dropped while one 9 below is kept; the cache
values are the Q8_0 values of the format oracle."""
import math

import numpy as np

import oracle
from oracle import attention as A


def _k_with_scores(q, targets, scale):
    """Keys whose scores against q (unit first element, zeros elsewhere) are the targets."""
    D = q.shape[0]
    K = np.zeros((len(targets), D))
    K[:, 0] = np.asarray(targets) / scale
    return K


def test_single_position_returns_its_value():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 128))
    K = rng.standard_normal((1, 128))
    V = rng.standard_normal((1, 128))
    out, _, kept = A.attention_f64(q, K, V, 0.1)
    assert np.array_equal(out[0], V[0]) and kept.all()


def test_two_positions_closed_form_weights():
    q = np.zeros((1, 128))
    q[0, 0] = 1.0
    K = _k_with_scores(q[0], [math.log(3.0), 0.0], 0.5)
    V = np.zeros((2, 128))
    V[0, :] = 4.0
    V[1, :] = -8.0
    out, s, _ = A.attention_f64(q, K, V, 0.5, skip_log=-math.inf)
    assert np.allclose(s[0], [math.log(3.0), 0.0], rtol=1e-15)
    assert np.allclose(out[0], 0.75 * 4.0 + 0.25 * -8.0, rtol=1e-14)


def test_equal_scores_give_the_mean():
    rng = np.random.default_rng(1)
    V = rng.standard_normal((7, 128))
    q = np.zeros((2, 128))
    K = np.zeros((7, 128))
    out, _, _ = A.attention_f64(q, K, V, 1.0)
    assert np.allclose(out, V.mean(axis=0), rtol=1e-13)


def test_skip_threshold_is_ln_1e_minus_4_below_the_max():
    q = np.zeros((1, 128))
    q[0, 0] = 1.0
    # scores 0 (the max), -9 (kept: above ln(1e-4) = -9.21), -10 (dropped)
    K = _k_with_scores(q[0], [0.0, -9.0, -10.0], 1.0)
    V = np.zeros((3, 128))
    V[0, 0], V[1, 0], V[2, 0] = 1.0, 2.0, 1000.0
    out, _, kept = A.attention_f64(q, K, V, 1.0)
    assert kept[0].tolist() == [True, True, False]
    w0, w1 = 1.0, math.exp(-9.0)
    assert math.isclose(out[0, 0], (w0 * 1.0 + w1 * 2.0) / (w0 + w1), rel_tol=1e-14)
    # without the threshold the dropped position contributes exp(-10) * 1000
    full, _, _ = A.attention_f64(q, K, V, 1.0, skip_log=-math.inf)
    w2 = math.exp(-10.0)
    assert math.isclose(full[0, 0], (w0 + 2 * w1 + 1000 * w2) / (w0 + w1 + w2), rel_tol=1e-14)
    assert math.isclose(A.SKIP_LOG, math.log(1e-4))


def test_grouped_heads_read_their_kv_head():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((4, 128))
    K = rng.standard_normal((2, 5, 128))
    V = rng.standard_normal((2, 5, 128))
    out = A.decode_attention_f64(q, K, V, 4, 0.09)
    for hq in range(4):
        ref = A.attention_f64(q[hq:hq + 1], K[hq // 2], V[hq // 2], 0.09)[0][0]
        assert np.allclose(out[hq], ref, rtol=1e-13, atol=1e-15)


def test_cache_values_are_q8_0():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 256)).astype(np.float32)
    v = A.q8_rows(x)
    assert np.array_equal(v, oracle.dequantize(oracle.Q8_0, oracle.quantize(oracle.Q8_0, x), 256))
    assert np.abs(v - x).max() <= np.abs(x).max() / 127
