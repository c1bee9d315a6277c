"""The dense decode step as the bench runs it (DenseDecoder: one epq_gemv_ex
call per matrix, weights streamed under programmatic dependent launch with
weights_ready, q/k/v read in place from the fused qkv buffer, the residual
stream updated in place) equals the same calls issued in isolation -- fresh
output buffers, a device synchronisation after each -- bit for bit, eagerly
and replayed from a CUDA graph.  The isolated calls are in turn checked
stage by stage against the float64 oracle (each op recomputed from the GPU's
own inputs, the method of "EPM ... 正確性"), at a small size and at the full
8B-class size (one layer and the 128256-row LM head, rows sampled).

The kernels are deterministic, so any difference between the chained step
and the isolated calls is a chaining hazard: an input read before its
producer's writes are visible, or an in-place update racing a reader.
"""
import numpy as np
import pytest
import torch

import oracle

from test_gpu_chain import Q4K, _Model

pytestmark = pytest.mark.gpu


class _Cfg:
    def __init__(self, m):
        self.layers, self.hidden, self.inter, self.vocab = m.L, m.H, m.I, m.V
        self.head_dim = m.hd
        self.kv_heads = m.nkv // m.hd
        self.heads = m.nq // m.hd
        self.rms_eps = m.eps

    @property
    def q_rows(self):
        return self.heads * self.head_dim

    @property
    def kv_rows(self):
        return self.kv_heads * self.head_dim


def _isolated(m, fmt):
    """Every op as its own epq_gemv_ex call into the model's distinct buffers."""
    e, H, nq, nkv = m.epq, m.H, m.nq, m.nkv
    h = m.x
    for l in range(m.L):
        W, B = m.W[l], m.buf[l]
        for buf in B.values():
            buf.fill_(float("nan"))
        e.epq_gemv_ex(fmt, W["qkv"], h, nq + 2 * nkv, H, y=B["qkv"], rms_prenorm=True, rms_eps=m.eps)
        torch.cuda.synchronize()
        e.epq_gemv_ex(fmt, W["o"], B["qkv"][:, nq + nkv:].contiguous(), H, nq, y=B["h1"], residual=h,
                      x_group=m.grp, x_head_dim=m.hd)
        torch.cuda.synchronize()
        e.epq_gemv_ex(fmt, W["gu"], B["h1"], 2 * m.I, H, y=B["m"], swiglu=True, rms_prenorm=True, rms_eps=m.eps)
        torch.cuda.synchronize()
        e.epq_gemv_ex(fmt, W["d"], B["m"], H, m.I, y=B["h2"], residual=B["h1"])
        torch.cuda.synchronize()
        h = B["h2"]
    m.logits.fill_(float("nan"))
    e.epq_gemv_ex(fmt, m.head, h, m.V, H, y=m.logits, rms_prenorm=True, rms_eps=m.eps)
    torch.cuda.synchronize()
    return m.logits.clone(), h.clone()


def _decoder_matches(m, ref_logits, ref_h):
    from moe_experts_gb300.decode import DenseDecoder
    cfg = _Cfg(m)
    layers = [(m.W[l]["qkv"], m.W[l]["o"], m.W[l]["gu"], m.W[l]["d"]) for l in range(m.L)]
    dec = DenseDecoder(cfg, Q4K, layers, m.head, m.dev, nvec=m.nvec)
    s = torch.cuda.Stream(device=m.dev)
    with torch.cuda.stream(s):
        for _ in range(2):                         # eager, back to back
            dec.step(m.x, stream=s)
    s.synchronize()
    assert torch.equal(dec.logits, ref_logits), "chained step differs from isolated calls (eager)"
    assert torch.equal(dec.h, ref_h)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dec.step(m.x, stream=s)
    for _ in range(3):
        dec.logits.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(dec.logits, ref_logits), "chained step differs from isolated calls (graph)"
    assert m.epq.epq_device_error() == 0


@pytest.mark.parametrize("nvec", [1, 2, 4, 8])
def test_dense_step_equals_isolated_calls(epq_lib, cuda_dev, nvec):
    m = _Model(epq_lib, cuda_dev, nvec, L=3, seed=11)
    logits, h = _isolated(m, Q4K)
    m.check()
    _decoder_matches(m, logits, h)


def test_dense_step_full_size_layer(epq_lib, cuda_dev):
    """One 8B-class layer (q 4096, k/v 1024, o 4096x4096, gate/up 2x14336,
    down 4096x14336) and the 128256-row LM head in the bench's launch
    configuration: stage-wise against the oracle on 128 sampled rows per op,
    and the chained step equal to the isolated calls bit for bit."""
    m = _Model(epq_lib, cuda_dev, 1, L=1, H=4096, nq=4096, nkv=1024, hd=128, I=14336, V=128256, seed=21)
    logits, h = _isolated(m, Q4K)
    m.check(rows_sample=128)
    _decoder_matches(m, logits, h)
    del m
    torch.cuda.empty_cache()


def test_dense_step_with_kv_attention_equals_isolated_calls(epq_lib, cuda_dev):
    """Attention mode (epq_attention_decode over a Q8_0 cache of 300
    positions between the qkv and o projections): the chained step equals
    the same calls issued in isolation, eagerly and from a CUDA graph."""
    import math
    from moe_experts_gb300.decode import SKIP_LOG, DenseDecoder
    m = _Model(epq_lib, cuda_dev, 1, L=2, seed=13, hd=128)
    cfg = _Cfg(m)
    layers = [(m.W[l]["qkv"], m.W[l]["o"], m.W[l]["gu"], m.W[l]["d"]) for l in range(m.L)]
    dec = DenseDecoder(cfg, Q4K, layers, m.head, m.dev, nvec=1, attn_ctx=300)
    e, H, nq, nkv = epq_lib, m.H, m.nq, m.nkv
    # isolated: fresh buffers, a synchronisation after every call
    h = m.x.clone()
    for l in range(m.L):
        W = m.W[l]
        qkv = e.epq_gemv_ex(Q4K, W["qkv"], h, nq + 2 * nkv, H, rms_prenorm=True, rms_eps=m.eps)
        torch.cuda.synchronize()
        att = e.epq_attention_decode(qkv[0, :nq].contiguous(), qkv[0, nq:nq + nkv].contiguous(),
                                     qkv[0, nq + nkv:].contiguous(), dec.caches[l], cfg.heads, 300,
                                     1.0 / math.sqrt(cfg.head_dim), SKIP_LOG)
        torch.cuda.synchronize()
        h1 = e.epq_gemv_ex(Q4K, W["o"], att.view(1, -1), H, nq, residual=h)
        torch.cuda.synchronize()
        mm = e.epq_gemv_ex(Q4K, W["gu"], h1, 2 * m.I, H, swiglu=True, rms_prenorm=True, rms_eps=m.eps)
        torch.cuda.synchronize()
        h = e.epq_gemv_ex(Q4K, W["d"], mm, H, m.I, residual=h1)
        torch.cuda.synchronize()
    ref = e.epq_gemv_ex(Q4K, m.head, h, m.V, H, rms_prenorm=True, rms_eps=m.eps)
    torch.cuda.synchronize()
    s = torch.cuda.Stream(device=m.dev)
    with torch.cuda.stream(s):
        dec.step(m.x, stream=s)
    s.synchronize()
    assert torch.equal(dec.logits, ref)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dec.step(m.x, stream=s)
    for _ in range(2):
        dec.logits.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(dec.logits, ref)
    assert epq_lib.epq_device_error() == 0
