"""GPU routing (softmax + top-K + grouping) against the oracle's selection
rule applied to the GPU's own float32 logits.

The top-K decision is taken on both sides from the same float32 logits, so
the selected experts must agree exactly (larger logit first, equal logits in
ascending expert order), for expert counts that are and are not multiples of
32, up to the 1024-expert maximum, and with exact ties.  Weights are checked
against the float64 softmax of those logits.  Expert weights are all-zero
blocks here (valid in every format), so the layer output must equal x
exactly: that checks that every token's entries reached the combine.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu


def _layer(epq, dev, E, H, I, R, bias=None, shared=False, norm=True, fmt=oracle.Q4_K):
    rb_h, rb_i = oracle.row_bytes(fmt, H), oracle.row_bytes(fmt, I)
    gu = torch.zeros((E, 2 * I, rb_h), dtype=torch.uint8, device=dev)
    dn = torch.zeros((E, H, rb_i), dtype=torch.uint8, device=dev)
    sgu = torch.zeros((2 * I, rb_h), dtype=torch.uint8, device=dev) if shared else None
    sdn = torch.zeros((H, rb_i), dtype=torch.uint8, device=dev) if shared else None
    rt = torch.from_numpy(np.ascontiguousarray(R, dtype=np.float32)).to(dev)
    bt = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).to(dev)
    return epq.MoELayer(fmt, rt, gu, dn, router_bias=bt, shared_gate_up=sgu, shared_down=sdn, norm_topk=norm)


def _route(epq, dev, layer, x, topk, stages):
    ntok = x.shape[0]
    xs = torch.from_numpy(x).to(dev)
    idx = torch.full((ntok, topk), -1, dtype=torch.int32, device=dev)
    w = torch.zeros((ntok, topk), dtype=torch.float32, device=dev)
    logits = torch.empty((ntok, layer.E), dtype=torch.float32, device=dev)
    y = torch.full_like(xs, float("nan"))
    epq.epq_moe_forward(layer, xs, topk, y=y, topk_idx=idx, topk_w=w, logits_out=logits, stages=stages)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy(), y.cpu().numpy()


def _check(idx, w, logits, topk, norm):
    ref_idx = oracle.topk_select(logits, topk)
    assert np.array_equal(idx, ref_idx), (idx[:2], ref_idx[:2])
    ref_w = oracle.combine_weights(logits, ref_idx, norm)
    # float32 softmax: the denominator sums <= 32 terms per lane, then a
    # 5-level butterfly (<= 37 roundings of a sum of terms in (0, 1]), each
    # term and the divisions within a few ulp: 1e-5 covers it
    assert np.allclose(w, ref_w, rtol=1e-5, atol=1e-12)


CASES = [  # E, H, topk, ntok
    (1, 256, 1, 1), (2, 256, 2, 3), (31, 512, 4, 2), (33, 256, 8, 1), (64, 1024, 6, 4),
    (256, 2048, 8, 1), (256, 2048, 8, 16), (1000, 512, 16, 5), (1024, 256, 10, 16), (16, 256, 16, 16),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("stages", [1, 0])   # routing kernel alone; full layer (routing inside gate/up)
def test_topk_matches_selection_rule(epq_lib, cuda_dev, case, stages):
    E, H, topk, ntok = case
    norm = (E + topk) % 2 == 0
    R = synthetic.student_t((E, H), seed=E * 7 + H).numpy()
    x = synthetic.normal((ntok, H), seed=E + ntok).numpy()
    layer = _layer(epq_lib, cuda_dev, E, H, 256, R, norm=norm, shared=(E % 2 == 1))
    idx, w, logits, y = _route(epq_lib, cuda_dev, layer, x, topk, stages)
    _check(idx, w, logits, topk, norm)
    if stages == 0:
        assert np.array_equal(y, x)           # zero experts: the combine adds exact zeros
    assert epq_lib.epq_device_error() == 0


def test_exact_ties_go_to_lower_expert(epq_lib, cuda_dev):
    E, H, topk = 300, 512, 5
    R = synthetic.student_t((E, H), seed=3).numpy()
    for e in (40, 77, 290, 299):       # bitwise-equal rows: bitwise-equal logits
        R[e] = R[11]
    bias = np.zeros(E, np.float32)
    bias[[11, 40, 77, 290, 299]] = 1e4
    x = synthetic.normal((2, H), seed=4).numpy()
    layer = _layer(epq_lib, cuda_dev, E, H, 256, R, bias=bias)
    for stages in (1, 0):
        idx, w, logits, _ = _route(epq_lib, cuda_dev, layer, x, topk, stages)
        assert (logits[:, [40, 77, 290, 299]] == logits[:, [11]]).all()
        assert idx.tolist() == [[11, 40, 77, 290, 299]] * 2
        assert np.allclose(w, 0.2, rtol=1e-6)


def test_all_equal_logits(epq_lib, cuda_dev):
    """A zero router: every logit is +0, the selection is experts 0..K-1."""
    E, H, topk, ntok = 96, 256, 7, 3
    layer = _layer(epq_lib, cuda_dev, E, H, 256, np.zeros((E, H), np.float32), norm=False)
    x = synthetic.normal((ntok, H), seed=1).numpy()
    idx, w, logits, _ = _route(epq_lib, cuda_dev, layer, x, topk, 0)
    assert idx.tolist() == [list(range(topk))] * ntok
    assert np.allclose(w, 1.0 / E, rtol=1e-6)


def test_workspace_needs_no_initialisation(epq_lib, cuda_dev):
    """A workspace full of 0xFF bytes gives the same layer output as a fresh
    one, on two calls in a row."""
    fmt, E, H, I, topk, ntok = oracle.Q4_0, 16, 512, 256, 4, 3
    R = synthetic.student_t((E, H), seed=21).numpy()
    gu = np.stack([oracle.quantize(fmt, synthetic.student_t((2 * I, H), seed=30 + e).numpy()) for e in range(E)])
    dn = np.stack([oracle.quantize(fmt, synthetic.student_t((H, I), seed=60 + e).numpy()) for e in range(E)])
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda_dev)
    layer = epq_lib.MoELayer(fmt, t(R), t(gu), t(dn))
    xs = t(synthetic.normal((ntok, H), seed=22).numpy())
    y0, _, _ = epq_lib.epq_moe_forward(layer, xs, topk)
    ws = torch.full((layer.workspace_bytes(ntok, topk),), 0xFF, dtype=torch.uint8, device=cuda_dev)
    for _ in range(2):
        y1, _, _ = epq_lib.epq_moe_forward(layer, xs, topk, workspace=ws)
        assert torch.equal(y0, y1)


@pytest.mark.parametrize("ntok,engine", [(2, 0), (4, 1)])
def test_stage_split_equals_single_call(epq_lib, cuda_dev, ntok, engine):
    """Router, gate/up and down issued as three calls give the single call's
    output bit for bit (the gate/up kernel routes from the stored logits).
    Same engine on both sides: two tokens on the tensor-core kernels, four
    on the CUDA-core ones (a single Q4_K call of more than two tokens would
    otherwise run in chunks of two on the tensor cores)."""
    prev = epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, engine)
    try:
        _stage_split(epq_lib, cuda_dev, ntok)
    finally:
        epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, prev)


def _stage_split(epq_lib, cuda_dev, ntok):
    fmt, E, H, I, topk = oracle.Q4_K, 24, 1024, 256, 3
    R = synthetic.student_t((E, H), seed=41).numpy()
    gu = np.stack([oracle.quantize(fmt, synthetic.student_t((2 * I, H), seed=50 + e).numpy()) for e in range(E)])
    dn = np.stack([oracle.quantize(fmt, synthetic.student_t((H, I), seed=90 + e).numpy()) for e in range(E)])
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda_dev)
    sgu = oracle.quantize(fmt, synthetic.student_t((2 * I, H), seed=42).numpy())
    sdn = oracle.quantize(fmt, synthetic.student_t((H, I), seed=43).numpy())
    layer = epq_lib.MoELayer(fmt, t(R), t(gu), t(dn), shared_gate_up=t(sgu), shared_down=t(sdn))
    xs = t(synthetic.normal((ntok, H), seed=44).numpy())
    y0, _, _ = epq_lib.epq_moe_forward(layer, xs, topk, rms_prenorm=True, rms_eps=1e-6)
    ws = torch.empty(layer.workspace_bytes(ntok, topk), dtype=torch.uint8, device=cuda_dev)
    y1 = torch.empty_like(xs)
    idx = torch.empty((ntok, topk), dtype=torch.int32, device=cuda_dev)
    for st in (1, 2, 4):
        epq_lib.epq_moe_forward(layer, xs, topk, y=y1, workspace=ws, rms_prenorm=True, rms_eps=1e-6, stages=st,
                                topk_idx=idx if st == 1 else None)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    assert (idx >= 0).all() and (idx < E).all()


@pytest.mark.parametrize("E,ties", [(200, (11, 40, 77, 190, 199)), (64, (0, 31, 32, 63)), (256, (5, 37, 69, 255))])
def test_one_token_ties_go_to_lower_expert(epq_lib, cuda_dev, E, ties):
    """One token (the single-warp selection for routers of up to 256
    experts): bitwise-equal logits in different lanes and in the same lane
    of the warp go to the lower expert, and an all-zero router selects
    experts 0..K-1."""
    H, topk = 512, len(ties)
    R = synthetic.student_t((E, H), seed=E + 9).numpy()
    for e in ties[1:]:
        R[e] = R[ties[0]]
    bias = np.zeros(E, np.float32)
    bias[list(ties)] = 1e4
    x = synthetic.normal((1, H), seed=E + 10).numpy()
    layer = _layer(epq_lib, cuda_dev, E, H, 256, R, bias=bias)
    for stages in (1, 0):
        idx, w, logits, _ = _route(epq_lib, cuda_dev, layer, x, topk, stages)
        assert idx.tolist() == [sorted(ties)]
        assert np.allclose(w, 1.0 / topk, rtol=1e-6)
    zero = _layer(epq_lib, cuda_dev, E, H, 256, np.zeros((E, H), np.float32), norm=False)
    idx, w, _, _ = _route(epq_lib, cuda_dev, zero, x, 7, 0)
    assert idx.tolist() == [list(range(7))]
    assert np.allclose(w, 1.0 / E, rtol=1e-6)
    assert epq_lib.epq_device_error() == 0
