"""GPU parity of the MoE layer (router + top-K + grouping, gate/up + SwiGLU,
down + weighted combine + residual) against the float64 oracle.

Acceptance (per token):
* top-K indices identical to the oracle's.  A token whose float64 margin
  between the K-th and (K+1)-th logit is within twice the router GEMV's
  error bound is "tie-ambiguous" (float32 rounding may legitimately swap
  the two); such inputs are never accepted silently: the input seed is
  replaced (deterministically) before anything runs on the GPU, the number
  of replacements is reported, and the test asserts that the inputs it
  finally runs have no ambiguous token;
* stage-wise, as in the EPM page's three-level verification: the SwiGLU
  outputs h (returned through h_out) against the oracle's on the same
  selection; then y against the oracle's down + combine fed with the GPU's
  own h and weights;
* end to end: |y - y_ref| <= 1e-3 (|x| + sum_k w_k A_k + g A_s).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle.moe import MoEWeights

pytestmark = pytest.mark.gpu
TOL = 1e-4


def _make(fmt, E, H, I, seed, shared=True, gate_vec=False, bias=False, norm=True, down_fmt=None):
    dfmt = fmt if down_fmt is None else down_fmt
    R = synthetic.student_t((E, H), seed=seed).numpy()
    gu = np.stack([oracle.quantize(fmt, synthetic.student_t((2 * I, H), seed=seed + 1 + e).numpy()) for e in range(E)])
    dn = np.stack([oracle.quantize(dfmt, synthetic.student_t((H, I), seed=seed + 1000 + e).numpy()) for e in range(E)])
    mw = MoEWeights(fmt=fmt, hidden=H, inter=I, router=R, gate_up=gu, down=dn, norm_topk=norm, down_fmt=down_fmt)
    if bias:
        mw.router_bias = synthetic.normal((E,), seed=seed + 5).numpy()
    if shared:
        mw.shared_gate_up = oracle.quantize(fmt, synthetic.student_t((2 * I, H), seed=seed + 7).numpy())
        mw.shared_down = oracle.quantize(dfmt, synthetic.student_t((H, I), seed=seed + 8).numpy())
        if gate_vec:
            mw.shared_gate_vec = synthetic.normal((H,), seed=seed + 9, scale=0.05).numpy()
    return mw


def _to_gpu(epq, mw, dev):
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return epq.MoELayer(mw.fmt, t(mw.router), t(mw.gate_up), t(mw.down), router_bias=t(mw.router_bias),
                        shared_gate_up=t(mw.shared_gate_up), shared_down=t(mw.shared_down),
                        shared_gate_vec=t(mw.shared_gate_vec), norm_topk=mw.norm_topk, down_fmt=mw.down_fmt)


def _run(epq, layer, x, topk, dev, rms_eps=None):
    ntok, H = x.shape
    xs = torch.from_numpy(x).to(dev)
    idx = torch.empty((ntok, topk), dtype=torch.int32, device=dev)
    w = torch.empty((ntok, topk), dtype=torch.float32, device=dev)
    h = torch.empty((ntok, topk + 1, layer.I), dtype=torch.float32, device=dev)
    logits = torch.empty((ntok, layer.E), dtype=torch.float32, device=dev)
    y, _, _ = epq.epq_moe_forward(layer, xs, topk, topk_idx=idx, topk_w=w, rms_prenorm=rms_eps is not None,
                                  rms_eps=rms_eps or 0.0, logits_out=logits, h_out=h)
    torch.cuda.synchronize()
    return (y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), h.cpu().numpy(), logits.cpu().numpy())


def _ambiguous_tokens(ref, topk, router):
    """Tokens whose K-th / (K+1)-th logit margin is within 2x the router
    GEMV bound 1e-4 * max_e sum_j |R_ej x_j| (float64 oracle logits)."""
    Abound = np.abs(ref.xin) @ np.abs(router.astype(np.float64)).T
    out = []
    for t in range(ref.logits.shape[0]):
        l = ref.logits[t]
        if topk >= l.size:
            continue
        order = np.argsort(-l, kind="stable")
        margin = l[order[topk - 1]] - l[order[topk]]
        if margin <= 2 * TOL * Abound[t].max():
            out.append(t)
    return out


def _unambiguous_inputs(mw, draw, topk, rms, tries=20):
    """Draw x with draw(attempt) until no token is tie-ambiguous; returns
    (x, oracle result, replacements)."""
    for attempt in range(tries):
        x = draw(attempt)
        ref = oracle.moe_forward_f64(mw, x, topk, rms_eps=rms)
        if not _ambiguous_tokens(ref, topk, mw.router):
            if attempt:
                print(f"tie-ambiguous input replaced {attempt} time(s)")
            return x, ref, attempt
    raise AssertionError("no unambiguous input found")


def _check_topk(ref, idx_gpu, topk, router):
    """Identical top-K; the inputs were chosen with no ambiguous token."""
    assert not _ambiguous_tokens(ref, topk, router)
    for t in range(idx_gpu.shape[0]):
        assert idx_gpu[t].tolist() == ref.idx[t].tolist(), (t, idx_gpu[t], ref.idx[t])


def _stagewise(mw, x, topk, idx, wts, h_gpu, y_gpu, xin, rms=False):
    """h vs oracle on the GPU's selection; y vs down+combine fed with h_gpu."""
    fmt, H, I = mw.fmt, mw.hidden, mw.inter
    dfmt = fmt if mw.down_fmt is None else mw.down_fmt
    ntok = x.shape[0]
    y_ref = x.astype(np.float64).copy()
    y_bound = 1e-6 * np.abs(x.astype(np.float64))
    for t in range(ntok):
        slots = [(k, int(idx[t, k])) for k in range(topk)]
        if mw.shared_gate_up is not None:
            slots.append((topk, -1))
        for k, e in slots:
            GU = mw.gate_up[e] if e >= 0 else mw.shared_gate_up
            D = mw.down[e] if e >= 0 else mw.shared_down
            gu = oracle.gemv_f64(fmt, GU, xin[t], H)[0]
            Agu = oracle.gemv_bound(fmt, GU, xin[t], H)[0]
            g, u, Ag, Au = gu[:I], gu[I:], Agu[:I], Agu[I:]
            silu = g / (1 + np.exp(-g))
            h_ref = silu * u
            hb = TOL * (1.1 * Ag * np.abs(u) + np.abs(silu) * Au) + 1e-6 * np.abs(h_ref) + 1e-30
            err = np.abs(h_gpu[t, k] - h_ref)
            assert (err <= hb).all(), f"h token {t} slot {k}: worst {(err / hb).max():.3g}"
            o = oracle.gemv_f64(dfmt, D, h_gpu[t, k], I)[0]
            Ao = oracle.gemv_bound(dfmt, D, h_gpu[t, k], I)[0]
            if e >= 0:
                wk = float(wts[t, k])
            elif mw.shared_gate_vec is not None:
                wk = 1 / (1 + np.exp(-(xin[t] @ mw.shared_gate_vec.astype(np.float64))))
            else:
                wk = 1.0
            y_ref[t] += wk * o
            y_bound[t] += abs(wk) * (TOL * Ao + 1e-6 * np.abs(o))
    err = np.abs(y_gpu - y_ref)
    assert (err <= y_bound + 1e-30).all(), f"combine: worst {(err / (y_bound + 1e-30)).max():.3g}"


def _end_to_end(mw, x, ref, y_gpu):
    fmt, H, I = mw.fmt, mw.hidden, mw.inter
    dfmt = fmt if mw.down_fmt is None else mw.down_fmt
    bound = np.abs(x.astype(np.float64)).copy()
    for t in range(x.shape[0]):
        slots = [(ref.w[t, k], mw.gate_up[e], mw.down[e]) for k, e in enumerate(ref.idx[t])]
        if mw.shared_gate_up is not None:
            gs = ref.shared_gate[t] if ref.shared_gate is not None else 1.0
            slots.append((gs, mw.shared_gate_up, mw.shared_down))
        for wk, GU, D in slots:
            _, g, u, h = oracle.expert_forward_f64(fmt, GU, D, H, I, ref.xin[t], mw.down_fmt)
            bound[t] += abs(wk) * oracle.gemv_bound(dfmt, D, h[0], I)[0]
    err = np.abs(y_gpu - ref.y)
    assert (err <= 1e-3 * bound).all(), f"end to end: worst {(err / (1e-3 * bound)).max():.3g}"


CASES = [
    # fmt, E, H, I, topk, ntok, shared, gate_vec, bias, norm, rms
    (oracle.Q4_K, 8, 512, 256, 2, 1, True, False, False, True, None),
    (oracle.Q4_K, 8, 512, 256, 2, 3, True, True, True, True, 1e-6),
    (oracle.Q8_0, 6, 256, 512, 3, 2, False, False, True, False, None),
    (oracle.Q4_0, 16, 1024, 256, 4, 8, True, False, False, True, 1e-5),
    (oracle.Q4_1, 5, 768, 256, 5, 4, True, True, False, True, None),
    (oracle.Q4_K, 32, 2048, 512, 8, 1, True, False, True, True, 1e-6),
    (oracle.Q4_K, 3, 256, 256, 1, 16, False, False, False, True, None),
]


@pytest.mark.parametrize("case", CASES)
def test_moe_parity(epq_lib, cuda_dev, case):
    _parity_case(epq_lib, cuda_dev, case)


# Q4_K with one or two tokens runs on the tensor-core expert kernels unless
# the CUDA-core engines are forced: both against the oracle.  Calls of more
# tokens route every token once, then run the expert stages in chunks of
# two (the logits, h and top-K outputs of every chunk checked).
TC_CASES = [
    # fmt, E, H, I, topk, ntok, shared, gate_vec, bias, norm, rms
    (oracle.Q4_K, 16, 1024, 512, 4, 1, True, True, True, True, 1e-6),
    (oracle.Q4_K, 16, 1024, 512, 4, 2, True, False, True, True, None),
    (oracle.Q4_K, 12, 1280, 768, 3, 2, True, False, False, False, 1e-5),  # 5 superblocks of x, 3 per h
    (oracle.Q4_K, 6, 256, 256, 6, 2, False, False, False, True, None),    # every expert chosen, no shared
    (oracle.Q4_K, 40, 4096, 256, 2, 1, True, False, False, True, None),   # slot boundaries inside stages
    # token chunks after one router launch for every token
    (oracle.Q4_K, 16, 1024, 512, 4, 5, True, True, True, True, 1e-6),
    (oracle.Q4_K, 40, 4096, 256, 2, 8, True, False, False, True, None),
]


@pytest.mark.parametrize("engine", [0, 1, 3])
@pytest.mark.parametrize("case", TC_CASES)
def test_moe_q4k_engines(epq_lib, cuda_dev, case, engine):
    prev = epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, engine)
    try:
        _parity_case(epq_lib, cuda_dev, case)
    finally:
        epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, prev)


# Q2_K / Q6_K experts (the 2-bit experts of "smolmaxxing") and mixed
# per-tensor recipes (the Q4_K gate/up + Q6_K down experts of "EPM ...
# 記憶體怎麼配置的"), each stage on its own engine: the k16 tensor-core
# kernels for Q2_K / Q6_K matrices, the Q4_K tensor-core or CUDA-core
# kernels for the other stage.
K16_CASES = [
    # fmt, down fmt, E, H, I, topk, ntok, shared, gate_vec, bias, norm, rms
    (oracle.Q2_K, None, 16, 1024, 512, 4, 1, True, True, True, True, 1e-6),
    (oracle.Q2_K, None, 16, 1024, 512, 4, 2, True, False, True, True, None),
    (oracle.Q6_K, None, 12, 1280, 768, 3, 2, True, False, False, False, 1e-5),  # odd superblock counts
    (oracle.Q6_K, None, 8, 512, 256, 2, 5, True, False, False, True, None),     # 5 tokens in chunks
    (oracle.Q4_K, oracle.Q6_K, 16, 1024, 512, 4, 1, True, False, True, True, None),
    (oracle.Q4_K, oracle.Q6_K, 16, 2048, 512, 8, 3, True, True, False, True, 1e-6),
    (oracle.Q2_K, oracle.Q4_K, 8, 512, 512, 2, 2, True, False, False, True, None),
    (oracle.Q8_0, oracle.Q2_K, 6, 256, 512, 3, 2, False, False, True, False, None),
    (oracle.Q6_K, oracle.Q8_0, 6, 512, 256, 2, 2, True, False, False, True, 1e-6),
    (oracle.Q2_K, None, 6, 256, 256, 6, 2, False, False, False, True, None),    # every expert chosen
]


@pytest.mark.parametrize("case", K16_CASES)
def test_moe_k16_formats_and_mixed(epq_lib, cuda_dev, case):
    fmt, dfmt = case[0], case[1]
    _parity_case(epq_lib, cuda_dev, (fmt,) + case[2:], down_fmt=dfmt)


@pytest.mark.parametrize("engine", [0, 1])
def test_moe_mixed_recipe_engines(epq_lib, cuda_dev, engine):
    """Q4_K gate/up with Q6_K down with the Q4_K stage on either engine."""
    prev = epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, engine)
    try:
        _parity_case(epq_lib, cuda_dev, (oracle.Q4_K, 16, 1024, 512, 4, 2, True, False, True, True, None),
                     down_fmt=oracle.Q6_K)
    finally:
        epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, prev)


def _parity_case(epq_lib, cuda_dev, case, down_fmt=None):
    fmt, E, H, I, topk, ntok, shared, gvec, bias, norm, rms = case
    mw = _make(fmt, E, H, I, seed=E * 100 + H + I + fmt, shared=shared, gate_vec=gvec, bias=bias, norm=norm,
               down_fmt=down_fmt)
    draw = lambda a: synthetic.normal((ntok, H), seed=H + ntok + 7919 * a, scale=2.0).numpy()
    x, ref, _ = _unambiguous_inputs(mw, draw, topk, rms)
    layer = _to_gpu(epq_lib, mw, cuda_dev)
    y, idx, w, h, logits = _run(epq_lib, layer, x, topk, cuda_dev, rms_eps=rms)
    # router logits within the GEMV bound
    Al = np.abs(ref.xin) @ np.abs(mw.router.astype(np.float64)).T
    assert (np.abs(logits - ref.logits) <= TOL * Al + 1e-6).all()
    _check_topk(ref, idx, topk, mw.router)
    assert np.allclose(w, ref.w, rtol=1e-4, atol=1e-6)
    _stagewise(mw, x, topk, idx, w, h, y, ref.xin)
    _end_to_end(mw, x, ref, y)
    assert epq_lib.epq_device_error() == 0


def test_moe_all_tokens_one_expert_and_inplace(epq_lib, cuda_dev):
    """A dominant router bias sends every token to expert 2 first; y may alias x."""
    fmt, E, H, I, topk, ntok = oracle.Q4_K, 8, 512, 256, 2, 5
    mw = _make(fmt, E, H, I, seed=77, shared=True)
    mw.router_bias = np.zeros(E, np.float32)
    mw.router_bias[2] = 1000.0
    x = synthetic.normal((ntok, H), seed=78).numpy()
    layer = _to_gpu(epq_lib, mw, cuda_dev)
    xs = torch.from_numpy(x).to(cuda_dev)
    idx = torch.empty((ntok, topk), dtype=torch.int32, device=cuda_dev)
    epq_lib.epq_moe_forward(layer, xs, topk, y=xs, topk_idx=idx)       # in place
    ref = oracle.moe_forward_f64(mw, x, topk)
    assert (idx.cpu().numpy()[:, 0] == 2).all()
    _end_to_end(mw, x, ref, xs.cpu().numpy())


def test_moe_zero_experts_identity_and_determinism(epq_lib, cuda_dev):
    fmt, E, H, I, topk, ntok = oracle.Q4_0, 4, 256, 256, 2, 3
    mw = _make(fmt, E, H, I, seed=5, shared=False)
    mw.gate_up = np.stack([oracle.quantize(fmt, np.zeros((2 * I, H), np.float32))] * E)
    mw.down = np.stack([oracle.quantize(fmt, np.zeros((H, I), np.float32))] * E)
    x = synthetic.normal((ntok, H), seed=6).numpy()
    layer = _to_gpu(epq_lib, mw, cuda_dev)
    y = _run(epq_lib, layer, x, topk, cuda_dev)[0]
    assert np.array_equal(y, x)
    mw2 = _make(oracle.Q4_K, 16, 512, 256, seed=9)
    layer2 = _to_gpu(epq_lib, mw2, cuda_dev)
    x2 = synthetic.normal((4, 512), seed=10).numpy()
    r1 = _run(epq_lib, layer2, x2, 4, cuda_dev)
    r2 = _run(epq_lib, layer2, x2, 4, cuda_dev)
    for a, b in zip(r1, r2):
        assert np.array_equal(a, b)


def test_moe_argument_errors(epq_lib, cuda_dev):
    mw = _make(oracle.Q4_K, 4, 256, 256, seed=3, shared=False)
    layer = _to_gpu(epq_lib, mw, cuda_dev)
    x = torch.zeros((1, 256), device=cuda_dev)
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_moe_forward(layer, x, 5)                             # topk > n_experts
    with pytest.raises(epq_lib.EpqError) as e:
        epq_lib.epq_moe_forward(layer, x, 2, workspace=torch.empty(16, dtype=torch.uint8, device=cuda_dev))
    assert e.value.status == 5
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_moe_forward(layer, torch.zeros((17, 256), device=cuda_dev), 2)   # ntok > 16


class _OraclePackedExperts:
    """Expert e's packed blocks, packed by the oracle on first use from the
    seeded float32 weights (the generator call the GPU side packed)."""

    def __init__(self, fmt, gen):
        self.fmt, self.gen, self.cache = fmt, gen, {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = oracle.quantize(self.fmt, self.gen(e).cpu().numpy())
        return self.cache[e]


@pytest.mark.parametrize("ntok", [1, 8])
def test_moe_full_size_layer(epq_lib, cuda_dev, ntok):
    """The single MoE layer at full size, in the bench's launch configuration:
    hidden 4096, 512 Q4_K experts of gate/up 2x1024x4096 + down 4096x1024
    (3.6 GB), a shared expert, router 512x4096 fp32, top-4; 1 and 8 tokens.
    Top-K against the oracle's, every selected expert stage-wise, and the
    GPU's packing of each selected expert bit-exact with the oracle's."""
    from synthetic import workloads as wl
    c = wl.MoELayer()
    H, I, E, K = c.hidden, c.inter, c.n_experts, c.topk
    fmt = oracle.Q4_K
    gen_gu = lambda e: wl.weight("moe_layer", 0, 10, 2 * I, H, cuda_dev, expert=e)
    gen_dn = lambda e: wl.weight("moe_layer", 0, 11, H, I, cuda_dev, expert=e)
    gu = torch.empty((E, 2 * I, epq_lib.epq_row_bytes(fmt, H)), dtype=torch.uint8, device=cuda_dev)
    dn = torch.empty((E, H, epq_lib.epq_row_bytes(fmt, I)), dtype=torch.uint8, device=cuda_dev)
    for e in range(E):
        epq_lib.epq_quantize(fmt, gen_gu(e), blocks=gu[e])
        epq_lib.epq_quantize(fmt, gen_dn(e), blocks=dn[e])
    R, _ = wl.moe_router("moe_layer", 0, E, H, cuda_dev, None)
    sgu_f = wl.weight("moe_layer", 0, 12, 2 * I, H, cuda_dev)
    sdn_f = wl.weight("moe_layer", 0, 13, H, I, cuda_dev)
    layer = epq_lib.MoELayer(fmt, R, gu, dn, shared_gate_up=epq_lib.epq_quantize(fmt, sgu_f),
                             shared_down=epq_lib.epq_quantize(fmt, sdn_f))
    mw = MoEWeights(fmt=fmt, hidden=H, inter=I, router=R.cpu().numpy(),
                    gate_up=_OraclePackedExperts(fmt, gen_gu), down=_OraclePackedExperts(fmt, gen_dn),
                    shared_gate_up=oracle.quantize(fmt, sgu_f.cpu().numpy()),
                    shared_down=oracle.quantize(fmt, sdn_f.cpu().numpy()))
    assert np.array_equal(mw.shared_gate_up, layer.shared_gate_up.cpu().numpy())
    draw = lambda a: wl.activations("moe_layer", ntok, H, cuda_dev, stream_id=a).cpu().numpy()
    x, ref, _ = _unambiguous_inputs(mw, draw, K, None)
    y, idx, w, h, logits = _run(epq_lib, layer, x, K, cuda_dev)
    Al = np.abs(ref.xin) @ np.abs(mw.router.astype(np.float64)).T
    assert (np.abs(logits - ref.logits) <= TOL * Al + 1e-6).all()
    _check_topk(ref, idx, K, mw.router)
    for e in sorted(set(idx.flatten().tolist())):
        assert np.array_equal(mw.gate_up[e], gu[e].cpu().numpy()), e
        assert np.array_equal(mw.down[e], dn[e].cpu().numpy()), e
    assert np.allclose(w, ref.w, rtol=1e-4, atol=1e-6)
    _stagewise(mw, x, K, idx, w, h, y, ref.xin)
    _end_to_end(mw, x, ref, y)
    assert epq_lib.epq_device_error() == 0
    del gu, dn
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fmt,dfmt", [(oracle.Q2_K, None), (oracle.Q4_K, oracle.Q6_K)])
def test_moe_full_size_decode_layer_k16(epq_lib, cuda_dev, fmt, dfmt):
    """One layer of the MoE decode model at full size with 2-bit experts and
    with the Q4_K + Q6_K-down recipe: hidden 2048, 256 experts of gate/up
    2x512x2048 + down 2048x512, a shared expert, top-8, one token.  Top-K
    against the oracle's, every selected expert stage-wise, and the GPU's
    packing of each selected expert bit-exact with the oracle's."""
    from synthetic import workloads as wl
    c = wl.MoEDecode()
    H, I, E, K = c.hidden, c.inter, c.n_experts, c.topk
    d = fmt if dfmt is None else dfmt
    gen_gu = lambda e: wl.weight("moe_decode", 0, 10, 2 * I, H, cuda_dev, expert=e)
    gen_dn = lambda e: wl.weight("moe_decode", 0, 11, H, I, cuda_dev, expert=e)
    gu = torch.empty((E, 2 * I, epq_lib.epq_row_bytes(fmt, H)), dtype=torch.uint8, device=cuda_dev)
    dn = torch.empty((E, H, epq_lib.epq_row_bytes(d, I)), dtype=torch.uint8, device=cuda_dev)
    for e in range(E):
        epq_lib.epq_quantize(fmt, gen_gu(e), blocks=gu[e])
        epq_lib.epq_quantize(d, gen_dn(e), blocks=dn[e])
    R, _ = wl.moe_router("moe_decode", 0, E, H, cuda_dev, None)
    sgu_f = wl.weight("moe_decode", 0, 12, 2 * I, H, cuda_dev)
    sdn_f = wl.weight("moe_decode", 0, 13, H, I, cuda_dev)
    layer = epq_lib.MoELayer(fmt, R, gu, dn, shared_gate_up=epq_lib.epq_quantize(fmt, sgu_f),
                             shared_down=epq_lib.epq_quantize(d, sdn_f), down_fmt=dfmt)
    mw = MoEWeights(fmt=fmt, hidden=H, inter=I, router=R.cpu().numpy(),
                    gate_up=_OraclePackedExperts(fmt, gen_gu), down=_OraclePackedExperts(d, gen_dn),
                    shared_gate_up=oracle.quantize(fmt, sgu_f.cpu().numpy()),
                    shared_down=oracle.quantize(d, sdn_f.cpu().numpy()), down_fmt=dfmt)
    assert np.array_equal(mw.shared_down, layer.shared_down.cpu().numpy())
    draw = lambda a: wl.activations("moe_decode", 1, H, cuda_dev, stream_id=a).cpu().numpy()
    x, ref, _ = _unambiguous_inputs(mw, draw, K, 1e-6)
    y, idx, w, h, logits = _run(epq_lib, layer, x, K, cuda_dev, rms_eps=1e-6)
    _check_topk(ref, idx, K, mw.router)
    for e in sorted(set(idx.flatten().tolist())):
        assert np.array_equal(mw.gate_up[e], gu[e].cpu().numpy()), e
        assert np.array_equal(mw.down[e], dn[e].cpu().numpy()), e
    assert np.allclose(w, ref.w, rtol=1e-4, atol=1e-6)
    _stagewise(mw, x, K, idx, w, h, y, ref.xin)
    _end_to_end(mw, x, ref, y)
    assert epq_lib.epq_device_error() == 0
    del gu, dn
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fmt,dfmt", [(oracle.Q2_K, None), (oracle.Q4_K, oracle.Q6_K)])
def test_moe_k16_stage_calls_equal_whole_call(epq_lib, cuda_dev, fmt, dfmt):
    """The router, gate/up and down stages issued by separate calls (one
    workspace) give the whole call's outputs bit for bit."""
    E, H, I, topk, ntok = 12, 1024, 512, 3, 2
    mw = _make(fmt, E, H, I, seed=606, shared=True, down_fmt=dfmt)
    layer = _to_gpu(epq_lib, mw, cuda_dev)
    x = torch.from_numpy(synthetic.normal((ntok, H), seed=607).numpy()).to(cuda_dev)
    ws = torch.empty(layer.workspace_bytes(ntok, topk), dtype=torch.uint8, device=cuda_dev)
    idx_a = torch.empty((ntok, topk), dtype=torch.int32, device=cuda_dev)
    y_a, _, _ = epq_lib.epq_moe_forward(layer, x, topk, topk_idx=idx_a, workspace=ws, rms_prenorm=True,
                                        rms_eps=1e-6)
    y_b = torch.empty_like(x)
    idx_b = torch.empty_like(idx_a)
    for st in (epq_lib.EPQ_MOE_ROUTE, epq_lib.EPQ_MOE_GATE_UP, epq_lib.EPQ_MOE_DOWN):
        epq_lib.epq_moe_forward(layer, x, topk, y=y_b, topk_idx=idx_b if st == epq_lib.EPQ_MOE_GATE_UP else None,
                                workspace=ws, rms_prenorm=True, rms_eps=1e-6, stages=st)
    torch.cuda.synchronize()
    assert torch.equal(idx_a, idx_b)
    assert torch.equal(y_a, y_b)
    assert epq_lib.epq_device_error() == 0


def test_moe_k16_argument_errors(epq_lib, cuda_dev):
    mw = _make(oracle.Q2_K, 8, 512, 256, seed=17, shared=False)
    layer = _to_gpu(epq_lib, mw, cuda_dev)
    x = torch.zeros((3, 512), device=cuda_dev)
    with pytest.raises(epq_lib.EpqError) as e:   # stage calls are not split into token chunks
        epq_lib.epq_moe_forward(layer, x, 2, stages=epq_lib.EPQ_MOE_GATE_UP)
    assert e.value.status == 3
    layer._x.down_fmt_set = 2                       # not 0 or 1
    with pytest.raises(epq_lib.EpqError) as e:
        epq_lib.epq_moe_forward(layer, x[:1], 2)
    assert e.value.status == 1
    layer._x.down_fmt_set, layer._x.down_fmt = 1, 9  # unknown format
    with pytest.raises(epq_lib.EpqError) as e:
        epq_lib.epq_moe_forward(layer, x[:1], 2)
    assert e.value.status == 2
