"""GPU parity of epq_attention_decode (decode attention over a Q8_0 key/value
cache with the skip threshold of the "smolmaxxing" compute table) against
the float64 oracle.

* the step's key and value rows land in the cache bit for bit as the format
  oracle's Q8_0 packs them (in the cache's factor-then-codes row order), and
  no other row changes;
* scores within 1e-5 * scale * sum_e |q_e k_e| of the float64 scores;
* the output against the oracle applied to the GPU's own float32 scores (the
  skip decision is then the same on both sides): within 1e-5 of
  sum_p w_p |v_p| / sum_p w_p per element;
* bitwise reproducible; cluster sizes 1 to 8, grouped heads 1 to 8, head
  sizes 128 and 256; score spreads with and without skipped positions;
* key/value rows copied in several shared-memory chunks (forced small
  chunks, and a long context of 8-head groups with 256-element heads whose
  scores leave room for chunks of ~90 rows only): the same bounds, and with
  chunks of 64 rows the output equals the one-chunk output bit for bit (the
  positions then fall to the same warps).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as A

pytestmark = pytest.mark.gpu


def _host_rows(x):
    """float32 [n, D] -> the cache rows [n, D + D/16]: the D/32 fp16 factors,
    then the D int8 codes of the oracle's Q8_0 blocks."""
    n, D = x.shape
    p = oracle.quantize(oracle.Q8_0, x).reshape(n, D // 32, 34)
    return np.concatenate([p[:, :, 0:2].reshape(n, -1), p[:, :, 2:].reshape(n, -1)], axis=1)


def _values(rows, D):
    """Cache rows -> float32 element values."""
    n = rows.shape[0]
    d = rows[:, :2 * (D // 32)].copy().view("<f2").astype(np.float32)          # [n, D/32]
    c = rows[:, 2 * (D // 32):].copy().view(np.int8).astype(np.float32)        # [n, D]
    return (c.reshape(n, D // 32, 32) * d[:, :, None]).reshape(n, D)


CASES = [
    # n_heads, n_kv, D, T (positions after the step), q spread
    (32, 8, 128, 1025, 1.0),
    (32, 8, 128, 1025, 4.0),
    (16, 16, 128, 300, 3.0),
    (8, 1, 256, 64, 2.0),
    (4, 2, 128, 1, 1.0),
    (16, 8, 128, 4000, 4.0),
    (8, 4, 256, 700, 5.0),
    (64, 8, 256, 12001, 3.0),
]


@pytest.mark.parametrize("case", CASES)
def test_attention_parity(epq_lib, cuda_dev, case):
    _check_case(epq_lib, cuda_dev, case)


@pytest.mark.parametrize("chunk", [8, 24, 64])
@pytest.mark.parametrize("case", [(32, 8, 128, 1025, 4.0), (8, 4, 256, 700, 5.0), (16, 16, 128, 300, 3.0)])
def test_attention_chunked_copies(epq_lib, cuda_dev, case, chunk):
    prev = epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_ATTN_CHUNK, chunk)
    try:
        out = _check_case(epq_lib, cuda_dev, case)
    finally:
        epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_ATTN_CHUNK, prev)
    if chunk == 64:
        assert torch.equal(out, _check_case(epq_lib, cuda_dev, case))


def _check_case(epq_lib, cuda_dev, case):
    n_heads, n_kv, D, T, spread = case
    rng = np.random.default_rng(T * 7 + D + n_heads)
    max_pos = T + 3
    Kf = rng.standard_normal((n_kv, T, D)).astype(np.float32)
    Vf = rng.standard_normal((n_kv, T, D)).astype(np.float32)
    q = (spread * rng.standard_normal((n_heads, D))).astype(np.float32)
    scale = 1.0 / math.sqrt(D)
    cache = epq_lib.KVCache(n_kv, D, max_pos, cuda_dev)
    hk = np.zeros((n_kv, max_pos, D + D // 16), np.uint8)
    hv = np.zeros_like(hk)
    hk[:, max_pos - 1] = 0x5A   # a row beyond the step that must not change
    for h in range(n_kv):
        hk[h, :T - 1] = _host_rows(Kf[h, :T - 1]) if T > 1 else hk[h, :0]
        hv[h, :T - 1] = _host_rows(Vf[h, :T - 1]) if T > 1 else hv[h, :0]
    cache.k.copy_(torch.from_numpy(hk))
    cache.v.copy_(torch.from_numpy(hv))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda_dev)
    k_new, v_new = Kf[:, T - 1], Vf[:, T - 1]
    out = torch.empty(n_heads * D, dtype=torch.float32, device=cuda_dev)
    scores = torch.full((n_heads, max_pos), float("nan"), dtype=torch.float32, device=cuda_dev)
    epq_lib.epq_attention_decode(t(q), t(k_new), t(v_new), cache, n_heads, T - 1, scale, A.SKIP_LOG, out=out,
                                 scores_out=scores)
    torch.cuda.synchronize()
    # the step's rows appended bit for bit, nothing else touched
    hk[:, T - 1] = _host_rows(k_new)
    hv[:, T - 1] = _host_rows(v_new)
    assert np.array_equal(cache.k.cpu().numpy(), hk)
    assert np.array_equal(cache.v.cpu().numpy(), hv)
    Kq = np.stack([_values(hk[h, :T], D) for h in range(n_kv)]).astype(np.float64)
    Vq = np.stack([_values(hv[h, :T], D) for h in range(n_kv)]).astype(np.float64)
    G = n_heads // n_kv
    s_gpu = scores.cpu().numpy()[:, :T].astype(np.float64)
    o_gpu = out.cpu().numpy().reshape(n_heads, D).astype(np.float64)
    kept_total = 0
    for h in range(n_kv):
        qh = q[h * G:(h + 1) * G].astype(np.float64)
        s_ref = scale * (qh @ Kq[h].T)
        mag = scale * (np.abs(qh) @ np.abs(Kq[h]).T)
        err = np.abs(s_gpu[h * G:(h + 1) * G] - s_ref)
        assert (err <= 1e-5 * mag + 1e-30).all(), f"scores head {h}: {(err / (1e-5 * mag + 1e-30)).max():.3g}"
        ref, _, kept = A.attention_f64(qh, Kq[h], Vq[h], scale, A.SKIP_LOG, scores=s_gpu[h * G:(h + 1) * G])
        kept_total += int(kept.sum())
        w = np.where(kept, np.exp(s_gpu[h * G:(h + 1) * G] - s_gpu[h * G:(h + 1) * G].max(1, keepdims=True)), 0)
        bound = 1e-5 * (w @ np.abs(Vq[h])) / w.sum(1, keepdims=True) + 1e-30
        e = np.abs(o_gpu[h * G:(h + 1) * G] - ref)
        assert (e <= bound).all(), f"output head {h}: {(e / bound).max():.3g}"
    assert 0 < kept_total <= n_heads * T
    if spread >= 4.0 and T > 100:
        assert kept_total < n_heads * T, "the case was meant to skip positions"
    # reproducible
    out2 = torch.empty_like(out)
    epq_lib.epq_attention_decode(t(q), t(k_new), t(v_new), cache, n_heads, T - 1, scale, A.SKIP_LOG, out=out2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    assert epq_lib.epq_device_error() == 0
    return out


def test_attention_step_by_step_append(epq_lib, cuda_dev):
    """Ten steps from an empty cache: each appends its row; the last output
    equals the oracle's (no threshold) on the accumulated cache."""
    n_heads, n_kv, D, T = 8, 4, 128, 10
    rng = np.random.default_rng(5)
    Kf = rng.standard_normal((T, n_kv, D)).astype(np.float32)
    Vf = rng.standard_normal((T, n_kv, D)).astype(np.float32)
    q = rng.standard_normal((T, n_heads, D)).astype(np.float32)
    cache = epq_lib.KVCache(n_kv, D, 16, cuda_dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda_dev)
    scale = 1.0 / math.sqrt(D)
    for p in range(T):
        out = epq_lib.epq_attention_decode(t(q[p]), t(Kf[p]), t(Vf[p]), cache, n_heads, p, scale, -math.inf)
    torch.cuda.synchronize()
    hk = cache.k.cpu().numpy()
    for h in range(n_kv):
        assert np.array_equal(hk[h, :T], _host_rows(Kf[:, h]))
    Kq = np.stack([_values(hk[h, :T], D) for h in range(n_kv)]).astype(np.float64)
    Vq = np.stack([_values(cache.v.cpu().numpy()[h, :T], D) for h in range(n_kv)]).astype(np.float64)
    ref = A.decode_attention_f64(q[T - 1].astype(np.float64), Kq, Vq, n_heads, scale, -math.inf)
    assert np.allclose(out.cpu().numpy().reshape(n_heads, D), ref, rtol=1e-4, atol=1e-5)


def test_attention_argument_errors(epq_lib, cuda_dev):
    cache = epq_lib.KVCache(2, 128, 8, cuda_dev)
    q = torch.zeros(6 * 128, device=cuda_dev)
    kv = torch.zeros(2 * 128, device=cuda_dev)
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_attention_decode(q, kv, kv, cache, 6, 0, 0.1)     # group 3
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_attention_decode(q[:512], kv, kv, cache, 4, 8, 0.1)   # pos >= max_pos
    with pytest.raises(ValueError):
        epq_lib.KVCache(2, 96, 8, cuda_dev)                               # head_dim 96
