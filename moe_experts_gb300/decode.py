"""Decode-step composition: the per-token sequence of library calls for a
dense 8B-class decoder and for a MoE decoder, ready to be captured in one
CUDA graph.

Each layer is pre-norm with a weightless RMS norm (folded into the GEMVs'
prologue).  Attention is either
* the one-token-context stand-in (attn_ctx=None): softmax over a single key
  is 1, so each query head's output is the value head it reads (grouped
  heads share one value head); q and k are still computed, so the weight
  traffic is that of a real decode step; or
* epq_attention_decode over a Q8_0 key/value cache per layer (attn_ctx = the
  number of cached positions before the step, filled with seeded synthetic
  keys and values): the step appends its key and value and attends over the
  cache with the ln(1e-4) skip threshold.
Every step below is one C-ABI call; this module holds device buffers and the
order of the calls, nothing else.

`timers` (optional) brackets each call of the first layer with a pair of
CUDA events, so that per-kernel durations can be read after a graph replay.
"""
from __future__ import annotations

import contextlib
import math

import torch

from . import _lib as L

SKIP_LOG = math.log(1e-4)


def kv_caches(n_layers, n_kv, head_dim, ctx, max_pos, device, seed):
    """One KVCache per layer with positions 0..ctx-1 filled: seeded N(0,1)
    keys and values quantized by epq_quantize (Q8_0) and laid out as the
    cache rows (block factors, then codes)."""
    gen = torch.Generator(device=device)
    caches = []
    nblk = head_dim // 32
    for li in range(n_layers):
        c = L.KVCache(n_kv, head_dim, max_pos, device)
        if ctx > 0:
            for dst in (c.k, c.v):
                gen.manual_seed(seed * 1000 + li * 2 + (dst is c.v))
                n = n_kv * ctx * head_dim
                x = torch.zeros(-(-n // 256) * 256, device=device, dtype=torch.float32)
                x[:n] = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
                # Q8_0 blocks are independent 32-runs: pack as rows of 256 and drop the padding
                b = L.epq_quantize(L.EPQ_Q8_0, x.view(-1, 256)).view(-1)[:n // 32 * 34].view(n_kv, ctx, nblk, 34)
                dst[:, :ctx, :2 * nblk] = b[..., :2].reshape(n_kv, ctx, 2 * nblk)
                dst[:, :ctx, 2 * nblk:] = b[..., 2:].reshape(n_kv, ctx, head_dim)
        caches.append(c)
    return caches


@contextlib.contextmanager
def _timed(timers, name, stream, on):
    if timers is None or not on:
        yield
        return
    a, b = timers.pair(name)
    a.record(stream)
    yield
    b.record(stream)


class DenseDecoder:
    """32-layer dense decoder + LM head, Q-format weights, nvec columns
    (one library call per matrix, or the whole step as one epq_gemv_chain).

    Per layer (h: [nvec, H] residual stream):
      qkv = Wqkv rms(h)                 (q, k, v rows concatenated)
      h   = h + Wo v                    (v heads repeated heads/kv_heads times)
      m   = silu(Wg rms(h)) * (Wu rms(h))
      h   = h + Wd m
    then logits = Whead rms(h).
    """

    def __init__(self, cfg, fmt, layers, head, device, nvec=1, chain=False, attn_ctx=None):
        self.cfg, self.fmt, self.layers, self.head, self.nvec = cfg, fmt, layers, head, nvec
        H = cfg.hidden
        self.qkv = torch.empty((nvec, cfg.q_rows + 2 * cfg.kv_rows), dtype=torch.float32, device=device)
        # KV-cache attention (one vector): caches of attn_ctx positions, the step at position attn_ctx
        self.attn_ctx = attn_ctx if (attn_ctx is not None and nvec == 1 and not chain) else None
        if self.attn_ctx is not None:
            self.caches = kv_caches(len(layers), cfg.kv_heads, cfg.head_dim, self.attn_ctx, self.attn_ctx + 64,
                                    device, seed=7)
            self.attn = torch.empty((1, cfg.q_rows), dtype=torch.float32, device=device)
            self.pos = self.attn_ctx
        self.m = torch.empty((nvec, cfg.inter), dtype=torch.float32, device=device)
        self.h = torch.empty((nvec, H), dtype=torch.float32, device=device)
        self.logits = torch.empty((nvec, cfg.vocab), dtype=torch.float32, device=device)
        # chain mode: the whole step is one epq_gemv_chain launch (Q4_K, nvec <= 2)
        self.chain = chain and fmt == L.EPQ_Q4_K and nvec <= 2
        self.ws = torch.zeros(L.epq_gemv_chain_workspace_bytes() if self.chain else 16, dtype=torch.uint8,
                              device=device)
        self._ops = {}

    def chain_ops(self, x):
        """The step's ops for epq_gemv_chain (same sequence as step())."""
        c, H = self.cfg, self.cfg.hidden
        nq, nkv = c.q_rows, c.kv_rows
        h = self.h
        ops = []
        for li, (wqkv, wo, wgu, wd) in enumerate(self.layers):
            src = x if li == 0 else h
            ops.append(L.gemv_op(wqkv, src, self.qkv, nq + 2 * nkv, H, rms_prenorm=True, rms_eps=c.rms_eps))
            ops.append(L.gemv_op(wo, self.qkv[:, nq + nkv:], h, H, nq, residual=src, x_group=c.heads // c.kv_heads,
                                 x_head_dim=c.head_dim))
            ops.append(L.gemv_op(wgu, h, self.m, 2 * c.inter, H, swiglu=True, rms_prenorm=True, rms_eps=c.rms_eps))
            ops.append(L.gemv_op(wd, self.m, h, H, c.inter, residual=h))
        ops.append(L.gemv_op(self.head, h, self.logits, c.vocab, H, rms_prenorm=True, rms_eps=c.rms_eps))
        return ops

    def step(self, x, stream=None, timers=None):
        """x [nvec, H] (read only) -> self.logits."""
        c, f, H = self.cfg, self.fmt, self.cfg.hidden
        if self.chain:
            key = x.data_ptr()
            if key not in self._ops:
                self._ops[key] = self.chain_ops(x)
            with _timed(timers, "gemv_chain", stream, True):
                L.epq_gemv_chain(f, self._ops[key], self.nvec, self.ws, stream=stream)
            return self.logits
        nq, nkv = c.q_rows, c.kv_rows
        h = self.h
        for li, (wqkv, wo, wgu, wd) in enumerate(self.layers):
            src = x if li == 0 else h
            on = li == 0
            with _timed(timers, "gemv_qkv", stream, on):
                L.epq_gemv_ex(f, wqkv, src, nq + 2 * nkv, H, y=self.qkv, rms_prenorm=True, rms_eps=c.rms_eps,
                              weights_ready=True, stream=stream)
            if self.attn_ctx is not None:
                q = self.qkv[0]
                L.epq_attention_decode(q[:nq], q[nq:nq + nkv], q[nq + nkv:], self.caches[li], c.heads, self.pos,
                                       1.0 / math.sqrt(c.head_dim), SKIP_LOG, out=self.attn[0], stream=stream)
                L.epq_gemv_ex(f, wo, self.attn, H, nq, y=h, residual=src, weights_ready=True, stream=stream)
            else:
                v = self.qkv[:, nq + nkv:]
                with _timed(timers, "gemv_o", stream, on):
                    L.epq_gemv_ex(f, wo, v, H, nq, y=h, residual=src, x_group=c.heads // c.kv_heads,
                                  x_head_dim=c.head_dim, weights_ready=True, stream=stream)
            with _timed(timers, "gemv_gateup", stream, on):
                L.epq_gemv_ex(f, wgu, h, 2 * c.inter, H, y=self.m, rms_prenorm=True, rms_eps=c.rms_eps,
                              swiglu=True, weights_ready=True, stream=stream)
            with _timed(timers, "gemv_down", stream, on):
                L.epq_gemv_ex(f, wd, self.m, H, c.inter, y=h, residual=h, weights_ready=True, stream=stream)
        L.epq_gemv_ex(f, self.head, h, c.vocab, H, y=self.logits, rms_prenorm=True, rms_eps=c.rms_eps,
                      weights_ready=True, stream=stream)
        return self.logits


class MoEDecoder:
    """MoE decoder, batch 1.

    Per layer: qkv = Wqkv rms(h); h = h + Wo v; h = h + MoE(rms(h)).
    """

    def __init__(self, cfg, fmt, layers, device, attn_ctx=None, max_new=64):
        self.cfg, self.fmt, self.layers = cfg, fmt, layers
        H = cfg.hidden
        self.qkv = torch.empty((1, 3 * H), dtype=torch.float32, device=device)
        self.h = torch.empty((1, H), dtype=torch.float32, device=device)
        # KV-cache attention (q, k and v each H = heads * head_dim: one key/value head per query head)
        self.attn_ctx = attn_ctx
        if attn_ctx is not None:
            self.caches = kv_caches(len(layers), cfg.heads, cfg.head_dim, attn_ctx, attn_ctx + max_new, device,
                                    seed=11)
            self.attn = torch.empty((1, H), dtype=torch.float32, device=device)
        ws = max(layer.workspace_bytes(1, cfg.topk) for (_, _, layer) in layers)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)

    def token(self, x, out, stream=None, timers=None, idx_out=None, pos=None):
        """x [1, H] (read only) -> out [1, H], the hidden state after the last layer.

        idx_out (optional, int32 [layers, topk]): each layer's selected experts.
        pos: the token's position in the key/value caches (attention mode)."""
        c, f, H = self.cfg, self.fmt, self.cfg.hidden
        h = self.h
        n = len(self.layers)
        for li, (wqkv, wo, moe) in enumerate(self.layers):
            src = x if li == 0 else h
            on = li == 0
            with _timed(timers, "gemv_qkv", stream, on):
                L.epq_gemv_ex(f, wqkv, src, 3 * H, H, y=self.qkv, rms_prenorm=True, rms_eps=c.rms_eps,
                              weights_ready=True, stream=stream)
            if self.attn_ctx is not None:
                q = self.qkv[0]
                L.epq_attention_decode(q[:H], q[H:2 * H], q[2 * H:], self.caches[li], c.heads, pos,
                                       1.0 / math.sqrt(c.head_dim), SKIP_LOG, out=self.attn[0], stream=stream)
                L.epq_gemv_ex(f, wo, self.attn, H, H, y=h, residual=src, weights_ready=True, stream=stream)
            else:
                with _timed(timers, "gemv_o", stream, on):
                    L.epq_gemv_ex(f, wo, self.qkv[:, 2 * H:], H, H, y=h, residual=src, weights_ready=True,
                                  stream=stream)
            y = out if li == n - 1 else h
            if timers is not None and on:
                for name, st in (("moe_router", L.EPQ_MOE_ROUTE), ("moe_gateup", L.EPQ_MOE_GATE_UP),
                                 ("moe_down", L.EPQ_MOE_DOWN)):
                    with _timed(timers, name, stream, True):
                        L.epq_moe_forward(moe, h, c.topk, y=y, workspace=self.ws, rms_prenorm=True,
                                          rms_eps=c.rms_eps, stages=st, stream=stream)
            else:
                L.epq_moe_forward(moe, h, c.topk, y=y, workspace=self.ws, rms_prenorm=True, rms_eps=c.rms_eps,
                                  topk_idx=None if idx_out is None else idx_out[li:li + 1], stream=stream)
        return out
