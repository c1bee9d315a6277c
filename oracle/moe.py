"""Mixture-of-experts layer oracle (test infrastructure only).

Follows "Flash-MoE：在笔记本上运行 397B 参数大模型": section "核心技术 /
3. Metal 计算着色器" lists the fused SwiGLU, the two-pass RMS norm and the
fused "combine + residual + sigmoid gate" kernel; section "每层流水线" runs
the router matvec, then softmax + top-K, then the K selected experts'
forward and the combine.  Expert shapes come from the same page (512
experts, K=4 plus a shared expert, hidden 4096) and from "EPM：
MiniCPM-V-4.7-35B-A3B 的 8 GiB 專家分頁 CPU 推論", section "記憶體怎麼配置的"
(256 experts, 8 per token).

Readings where the pages are silent (listed in the design notes):

* Selection is top-K on the router logits (softmax is monotone, so this is
  the same set as top-K on probabilities); equal logits go to the lower
  expert index.
* Softmax runs over all E logits with the maximum subtracted.  With
  ``norm_topk`` the K selected probabilities are divided by their sum;
  without it they are used as they are.
* An expert is ``down( silu(gate x) * (up x) )`` with
  ``silu(g) = g / (1 + exp(-g))``.  The packed gate/up matrix of an expert
  holds the ``inter`` gate rows followed by the ``inter`` up rows.
* The shared expert (optional) enters with weight 1, or with
  ``sigmoid(g_s . x)`` when a gate vector is given.
* ``y = x + sum_k w_k o_k + g_s o_shared``.  With ``rms_eps`` set, the router
  and all experts see ``x / sqrt(mean(x^2) + eps)`` while the residual stays
  ``x`` (a weightless pre-norm, the decode-step configuration).

Everything is float64 except the stored weights, which enter through the
format oracle's dequantizer.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .formats import dequantize


def rmsnorm_f64(x: np.ndarray, eps: float) -> np.ndarray:
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + float(np.float32(eps)))


def router_logits_f64(R: np.ndarray, x: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    """R float32 [E, H], x [ntok, H] -> logits float64 [ntok, E]."""
    l = np.asarray(x, np.float64) @ np.asarray(R, np.float64).T
    if bias is not None:
        l = l + np.asarray(bias, np.float64)
    return l


def topk_select(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per row, largest first; ties -> lower index."""
    logits = np.atleast_2d(logits)
    out = np.empty((logits.shape[0], k), np.int32)
    for t in range(logits.shape[0]):
        order = sorted(range(logits.shape[1]), key=lambda e: (-logits[t, e], e))
        out[t] = order[:k]
    return out


def softmax_f64(logits: np.ndarray) -> np.ndarray:
    l = np.atleast_2d(np.asarray(logits, np.float64))
    e = np.exp(l - l.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def combine_weights(logits: np.ndarray, idx: np.ndarray, norm_topk: bool) -> np.ndarray:
    p = softmax_f64(logits)
    w = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    if norm_topk:
        w = w / w.sum(axis=1, keepdims=True)
    return w


def silu_f64(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def expert_forward_f64(fmt: int, gate_up: np.ndarray, down: np.ndarray,
                       hidden: int, inter: int, x: np.ndarray, down_fmt: int | None = None):
    """One expert on x [n, hidden] -> (o [n, hidden], g, u, h [n, inter]).
    down_fmt: the down matrix's format when it differs from fmt."""
    GU = dequantize(fmt, gate_up, hidden).astype(np.float64)     # [2*inter, hidden]
    D = dequantize(fmt if down_fmt is None else down_fmt, down, inter).astype(np.float64)   # [hidden, inter]
    x = np.atleast_2d(np.asarray(x, np.float64))
    g = x @ GU[:inter].T
    u = x @ GU[inter:].T
    h = silu_f64(g) * u
    return h @ D.T, g, u, h


@dataclass
class MoEWeights:
    """Packed expert weights as the library stores them.

    gate_up: uint8 [E, 2*inter, row_bytes(hidden)]; down: uint8
    [E, hidden, row_bytes(inter)]; router: float32 [E, hidden].  down_fmt:
    the down projections' format in a mixed per-tensor recipe (the Q6_K
    ffn_down_exps next to Q4_K gate/up of "EPM ... 記憶體怎麼配置的"); None =
    fmt.
    """
    fmt: int
    hidden: int
    inter: int
    router: np.ndarray
    gate_up: np.ndarray
    down: np.ndarray
    router_bias: np.ndarray | None = None
    shared_gate_up: np.ndarray | None = None
    shared_down: np.ndarray | None = None
    shared_gate_vec: np.ndarray | None = None
    norm_topk: bool = True
    down_fmt: int | None = None

    @property
    def n_experts(self) -> int:
        return self.router.shape[0]


@dataclass
class MoEResult:
    y: np.ndarray                  # [ntok, hidden]
    idx: np.ndarray                # [ntok, K] int32
    w: np.ndarray                  # [ntok, K] combine weights
    logits: np.ndarray             # [ntok, E]
    xin: np.ndarray                # [ntok, hidden] what router and experts saw
    shared_gate: np.ndarray | None = None          # [ntok]
    stages: dict = field(default_factory=dict)     # (t, slot) -> (g, u, h, o)


def moe_forward_f64(mw: MoEWeights, x: np.ndarray, topk: int,
                    rms_eps: float | None = None, keep_stages: bool = False) -> MoEResult:
    x = np.atleast_2d(np.asarray(x, np.float32))
    x64 = x.astype(np.float64)
    xin = rmsnorm_f64(x64, rms_eps) if rms_eps is not None else x64
    logits = router_logits_f64(mw.router, xin, mw.router_bias)
    idx = topk_select(logits, topk)
    w = combine_weights(logits, idx, mw.norm_topk)
    y = x64.copy()
    stages = {}
    gs = None
    for t in range(x.shape[0]):
        for slot in range(topk):
            e = int(idx[t, slot])
            o, g, u, h = expert_forward_f64(mw.fmt, mw.gate_up[e], mw.down[e],
                                            mw.hidden, mw.inter, xin[t], mw.down_fmt)
            y[t] += w[t, slot] * o[0]
            if keep_stages:
                stages[(t, slot)] = (g[0], u[0], h[0], o[0])
    if mw.shared_gate_up is not None:
        if mw.shared_gate_vec is not None:
            gs = 1.0 / (1.0 + np.exp(-(xin @ np.asarray(mw.shared_gate_vec, np.float64))))
        else:
            gs = np.ones(x.shape[0])
        for t in range(x.shape[0]):
            o, g, u, h = expert_forward_f64(mw.fmt, mw.shared_gate_up, mw.shared_down,
                                            mw.hidden, mw.inter, xin[t], mw.down_fmt)
            y[t] += gs[t] * o[0]
            if keep_stages:
                stages[(t, topk)] = (g[0], u[0], h[0], o[0])
    return MoEResult(y=y, idx=idx, w=w, logits=logits, xin=xin, shared_gate=gs, stages=stages)
