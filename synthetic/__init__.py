"""Seeded synthetic inputs shared by the tests, the bench and the checker.

This module only draws numbers.  It holds none of the quantization, GEMV or
mixture-of-experts arithmetic: both the CUDA path and the CPU oracle receive
what is drawn here as plain input tensors.

Distributions follow the workloads the source pages describe:

* weights: Student-t with 5 degrees of freedom times 0.02 (the long-tailed
  sample of the edge-inference handbook page, "GGUF quantization formats"
  section), drawn as ``Z / sqrt(chi2_5 / 5)`` with ``chi2_5`` the sum of five
  squared standard normals;
* activations: standard normal;
* router bias for Zipf-like expert popularity: ``-s * ln(rank(e))`` with a
  seeded permutation for ``rank`` (the construction is stated with the
  decode-step workload in the design notes).

Every generator takes an explicit integer seed and an optional torch device;
the same seed on the same device always gives the same tensor.
"""
from __future__ import annotations

import math

import torch

STUDENT_T_DF = 5
WEIGHT_SCALE = 0.02


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def mix_seed(*parts: int) -> int:
    """splitmix64 over the parts: one seed per (config, layer, tensor)."""
    z = 0x9E3779B97F4A7C15
    for p in parts:
        z = (z + (int(p) & 0xFFFF_FFFF_FFFF_FFFF) + 0x9E3779B97F4A7C15) & 0xFFFF_FFFF_FFFF_FFFF
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFF_FFFF_FFFF_FFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFF_FFFF_FFFF_FFFF
        z ^= z >> 31
    return z & 0x7FFF_FFFF_FFFF_FFFF


def student_t(shape, seed: int, scale: float = WEIGHT_SCALE, device="cpu") -> torch.Tensor:
    """float32 Student-t(5) * scale, drawn as Z / sqrt(chi2_5 / 5)."""
    g = _gen(seed, device)
    shape = tuple(shape)
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(STUDENT_T_DF):
        n = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        chi2.addcmul_(n, n)
    t = z / torch.sqrt(chi2 / STUDENT_T_DF)
    return (t * scale).contiguous()


def normal(shape, seed: int, scale: float = 1.0, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return (torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32) * scale).contiguous()


def uniform_int(shape, low: int, high: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randint(low, high, tuple(shape), generator=g, device=device, dtype=torch.int64)


def page2_sample() -> torch.Tensor:
    """The handbook page's own 1M-weight sample: torch's global seed 0, then
    1,048,576 draws of torch's Student-t(5) sampler, times 0.02.

    Used only to pin the oracle to the relative errors the page prints.
    """
    torch.manual_seed(0)
    return (torch.distributions.StudentT(5.0).sample((4096 * 256,)) * 0.02).contiguous()


def zipf_router_bias(n_experts: int, seed: int, s: float = 1.1) -> torch.Tensor:
    """Additive router bias -s*ln(rank(e)) with a seeded rank permutation.

    With router logits of Gumbel spread (std pi/sqrt(6)), top-k over
    logits + bias approximates sampling experts with probability
    proportional to rank**-s.
    """
    g = _gen(seed, "cpu")
    perm = torch.randperm(n_experts, generator=g)
    rank = torch.empty(n_experts, dtype=torch.float64)
    rank[perm] = torch.arange(1, n_experts + 1, dtype=torch.float64)
    return (-s * torch.log(rank)).to(torch.float32)


GUMBEL_STD = math.pi / math.sqrt(6.0)
