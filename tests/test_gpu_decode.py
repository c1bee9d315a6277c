"""The chained decode path equals isolated calls bit for bit.

MoEDecoder issues every layer's calls back to back on one stream (each
kernel starts under programmatic dependent launch while the previous one
drains), reuses its activation buffers and one MoE workspace across layers,
and runs here inside a CUDA graph as the bench does.  The same computation
issued as isolated calls -- fresh output buffers and a fresh workspace for
every call, a device synchronisation after each -- must give the same bits:
the kernels are deterministic, so any difference is a chaining hazard (a
read before the producer's writes are visible, stale cached lines, a
workspace overwritten too early).  Each isolated call is checked against the
oracle by the other GPU tests.
"""
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu


class _Cfg:
    hidden, n_experts, inter, topk, rms_eps = 512, 16, 256, 4, 1e-6


def _model(epq, dev, nl, fmt):
    c = _Cfg
    H, E, I = c.hidden, c.n_experts, c.inter
    layers = []
    for l in range(nl):
        q = lambda rows, cols, tid: epq.epq_quantize(fmt, synthetic.student_t((rows, cols), seed=1000 * l + tid,
                                                                              scale=0.05, device=dev))
        wqkv, wo = q(3 * H, H, 1), q(H, H, 2)
        R = synthetic.student_t((E, H), seed=1000 * l + 3, scale=0.1, device=dev)
        gu = torch.stack([q(2 * I, H, 10 + e) for e in range(E)])
        dn = torch.stack([q(H, I, 100 + e) for e in range(E)])
        layer = epq.MoELayer(fmt, R, gu, dn, shared_gate_up=q(2 * I, H, 4), shared_down=q(H, I, 5))
        layers.append((wqkv, wo, layer))
    return layers


def _isolated_token(epq, layers, x, fmt):
    c, H = _Cfg, _Cfg.hidden
    h = x.clone()
    for wqkv, wo, moe in layers:
        qkv = epq.epq_gemv_ex(fmt, wqkv, h, 3 * H, H, rms_prenorm=True, rms_eps=c.rms_eps)
        torch.cuda.synchronize()
        h2 = epq.epq_gemv_ex(fmt, wo, qkv[:, 2 * H:].contiguous(), H, H, residual=h)
        torch.cuda.synchronize()
        ws = torch.empty(moe.workspace_bytes(1, c.topk), dtype=torch.uint8, device=x.device)
        h, _, _ = epq.epq_moe_forward(moe, h2, c.topk, workspace=ws, rms_prenorm=True, rms_eps=c.rms_eps)
        torch.cuda.synchronize()
    return h


@pytest.mark.parametrize("fmt", [oracle.Q4_K, oracle.Q8_0])
def test_chained_decode_equals_isolated_calls(epq_lib, cuda_dev, fmt):
    from moe_experts_gb300.decode import MoEDecoder
    nl, ntoks = 3, 3
    layers = _model(epq_lib, cuda_dev, nl, fmt)
    xs = synthetic.normal((ntoks, _Cfg.hidden), seed=77, device=cuda_dev)
    ref = torch.cat([_isolated_token(epq_lib, layers, xs[t:t + 1], fmt) for t in range(ntoks)])

    model = MoEDecoder(_Cfg, fmt, layers, cuda_dev)
    out = torch.empty_like(xs)
    s = torch.cuda.Stream(device=cuda_dev)
    with torch.cuda.stream(s):
        for t in range(ntoks):                       # eager, chained
            model.token(xs[t:t + 1], out[t:t + 1], stream=s)
    s.synchronize()
    assert torch.equal(out, ref)

    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for t in range(ntoks):
            model.token(xs[t:t + 1], out[t:t + 1], stream=s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert epq_lib.epq_device_error() == 0


def test_layers_interleaved_on_one_workspace(epq_lib, cuda_dev):
    """Two different MoE layers alternating on one workspace without host
    synchronisation give what each gives alone."""
    fmt = oracle.Q4_K
    layers = _model(epq_lib, cuda_dev, 2, fmt)
    A, B = layers[0][2], layers[1][2]
    xs = synthetic.normal((6, _Cfg.hidden), seed=5, device=cuda_dev)
    ref = []
    for i in range(6):
        y, _, _ = epq_lib.epq_moe_forward(A if i % 2 == 0 else B, xs[i:i + 1], 4)
        torch.cuda.synchronize()
        ref.append(y)
    ws = torch.empty(max(A.workspace_bytes(1, 4), B.workspace_bytes(1, 4)), dtype=torch.uint8, device=cuda_dev)
    out = torch.empty_like(xs)
    for i in range(6):
        epq_lib.epq_moe_forward(A if i % 2 == 0 else B, xs[i:i + 1], 4, y=out[i:i + 1], workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, torch.cat(ref))
