"""Seeded synthetic workloads: shapes, seeds and value laws of the decode
configurations (no quantization or GEMV arithmetic here).

* ``gemv4096``   single Q4_K dequant-GEMV, W 4096x4096, x ~ N(0,1)
* ``layer8b``    one dense 8B-class decoder layer: q 4096x4096, k/v 1024x4096,
                 o 4096x4096, gate/up 14336x4096, down 4096x14336 (per format)
* ``dense8b``    32 such layers + LM head 128256x4096, batch 1 and nvec 2/4/8
* ``moe_layer``  hidden 4096, 512 experts of gate/up 1024x4096 + down
                 4096x1024, one shared expert, router 512x4096 fp32, top-4,
                 1 and 8 tokens
* ``moe_decode`` 40 layers, hidden 2048, 256 experts of gate/up 512x2048 +
                 down 2048x512, top-8 + shared, attention q/k/v/o 2048x2048,
                 router 256x2048 with Zipf(1.1) expert popularity, a 64-token
                 decode run at batch 1

Weights are Student-t(5) * 0.02 (the handbook page's sample law); the
router of ``moe_decode`` is scaled so that its logits have the Gumbel
standard deviation pi/sqrt(6) on unit-RMS inputs, and its additive bias is
-1.1 ln rank(e) with a seeded rank permutation per layer: top-8 then draws
experts roughly like Plackett-Luce sampling proportional to rank^-1.1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

from . import GUMBEL_STD, mix_seed, normal, student_t, zipf_router_bias

CONFIG_IDS = {"gemv4096": 1, "layer8b": 2, "dense8b": 3, "moe_layer": 4, "moe_decode": 5}


@dataclass(frozen=True)
class DenseDecode:
    layers: int = 32
    hidden: int = 4096
    heads: int = 32
    kv_heads: int = 8
    head_dim: int = 128
    inter: int = 14336
    vocab: int = 128256
    rms_eps: float = 1e-5

    @property
    def q_rows(self):
        return self.heads * self.head_dim

    @property
    def kv_rows(self):
        return self.kv_heads * self.head_dim


@dataclass(frozen=True)
class MoEDecode:
    layers: int = 40
    hidden: int = 2048
    heads: int = 16
    head_dim: int = 128
    n_experts: int = 256
    inter: int = 512
    topk: int = 8
    tokens: int = 64
    zipf_s: float = 1.1
    rms_eps: float = 1e-6


@dataclass(frozen=True)
class MoELayer:
    hidden: int = 4096
    n_experts: int = 512
    inter: int = 1024
    topk: int = 4


def weight(cfg: str, layer: int, tensor: int, rows: int, cols: int, device, expert: int = 0, scale: float = 0.02):
    """float32 [rows, cols] Student-t(5)*scale for one tensor of a config."""
    return student_t((rows, cols), seed=mix_seed(CONFIG_IDS[cfg], layer, tensor, expert), scale=scale,
                     device=device)


def activations(cfg: str, n: int, cols: int, device, stream_id: int = 0):
    return normal((n, cols), seed=mix_seed(CONFIG_IDS[cfg], 999_999, stream_id), device=device)


def moe_router(cfg: str, layer: int, n_experts: int, hidden: int, device, zipf_s: float | None):
    """Router weights (and Zipf bias when zipf_s is given) of one layer."""
    if zipf_s is None:
        return weight(cfg, layer, 50, n_experts, hidden, device), None
    # Student-t(5) has variance 5/3: scale so that std(R x) = pi/sqrt(6) for unit-RMS x
    s = GUMBEL_STD / math.sqrt(hidden * 5.0 / 3.0)
    R = weight(cfg, layer, 50, n_experts, hidden, device, scale=s)
    b = zipf_router_bias(n_experts, seed=mix_seed(CONFIG_IDS[cfg], layer, 51), s=zipf_s).to(device)
    return R, b
