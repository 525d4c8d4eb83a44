"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module draws random numbers and rounds them to bf16; it holds none of the
codec's arithmetic. Every generator takes a seed and a torch device and returns
a torch tensor of bf16 *bit patterns* (dtype int16, reinterpret as uint16).
The same seed on the same device always gives the same tensor; CPU and CUDA
generators differ, so a test that needs the oracle and the GPU to see the same
values draws on one device and copies.

Workload shapes follow the Cassandra paper's evaluation models (Llama-3-8B,
Qwen3-8B decoder stacks, their KV caches); weights and activations are
synthetic stand-ins, since no checkpoint or dataset is used.
"""
from __future__ import annotations

import math

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def to_bits(t: torch.Tensor) -> torch.Tensor:
    """float tensor -> bf16 (round to nearest even) -> int16 bit pattern."""
    return t.to(torch.bfloat16).view(torch.int16)


def normal_weight(N: int, K: int, seed: int, std: float = 0.02, outlier_frac: float = 0.0,
                  outlier_mul: float = 20.0, device="cpu") -> torch.Tensor:
    """W ~ N(0, std); a fraction of entries (picked by a random permutation of
    the same generator) multiplied by outlier_mul."""
    g = _gen(seed, device)
    w = torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * std
    n_out = int(round(outlier_frac * N * K))
    if n_out:
        idx = torch.randperm(N * K, generator=g, device=device)[:n_out]
        w.view(-1)[idx] *= outlier_mul
    return to_bits(w)


def t4_weight(N: int, K: int, seed: int, std: float = 0.02, device="cpu") -> torch.Tensor:
    """W = std * t4 / sqrt(2): Student-t with 4 degrees of freedom scaled to
    standard deviation std (t4 has variance 2). t4 = z / sqrt(chi2_4 / 4)."""
    g = _gen(seed, device)
    w = torch.empty(N, K, device=device, dtype=torch.float32)
    rows = max(1, (1 << 24) // max(K, 1))  # bounded temporaries
    for r0 in range(0, N, rows):
        r1 = min(N, r0 + rows)
        z = torch.randn(5, r1 - r0, K, generator=g, device=device, dtype=torch.float32)
        chi = (z[1:] ** 2).sum(0) / 4.0
        w[r0:r1] = z[0] / chi.sqrt() * (std / math.sqrt(2.0))
    return to_bits(w)


def activations(nvec: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """x ~ N(0, 1), [nvec][K]."""
    g = _gen(seed, device)
    return to_bits(torch.randn(nvec, K, generator=g, device=device, dtype=torch.float32))


def kv_channel_scale(seed: int, D: int = 128, device="cpu") -> torch.Tensor:
    """Per-channel scale ~ LogNormal(0, 0.5), drawn once per (layer, head, K|V)."""
    g = _gen(seed, device)
    return torch.exp(0.5 * torch.randn(D, generator=g, device=device, dtype=torch.float32))


def kv_tokens(T: int, H: int, seed: int, scales: torch.Tensor, D: int = 128, device="cpu") -> torch.Tensor:
    """K or V for T tokens and H kv heads: N(0,1) * scale[h][channel], [T][H][D].
    scales is [H][D]."""
    g = _gen(seed, device)
    x = torch.randn(T, H, D, generator=g, device=device, dtype=torch.float32)
    return to_bits(x * scales.to(device)[None, :, :])


def kv_scales(layer: int, H: int, which: int, D: int = 128, device="cpu") -> torch.Tensor:
    """[H][D] channel scales of one layer's K (which=0) or V (which=1)."""
    return torch.stack([kv_channel_scale(1_000_003 * layer + 7919 * h + which, D, device) for h in range(H)])


def cfg0_weight(device="cpu") -> torch.Tensor:
    """Single 4096x4096 matrix, N(0, 0.02) with 0.1% outliers x20, seed 0."""
    return normal_weight(4096, 4096, seed=0, std=0.02, outlier_frac=0.001, outlier_mul=20.0, device=device)


# Llama-3-8B: 32 layers, hidden 4096, FFN 14336, 32 q heads / 8 kv heads of 128,
# vocabulary 128256, rotary base 500000.
LLAMA3_8B = dict(layers=32, hidden=4096, ffn=14336, n_q=32, n_kv=8, head_dim=128, vocab=128256,
                 rope_theta=500000.0)
# Qwen3-8B: 36 layers, hidden 4096, FFN 12288, 32/8 heads, vocabulary 151936,
# rotary base 1000000.
QWEN3_8B = dict(layers=36, hidden=4096, ffn=12288, n_q=32, n_kv=8, head_dim=128, vocab=151936,
                rope_theta=1000000.0)


def norm_weight(dim: int, seed: int, device="cpu") -> torch.Tensor:
    """RMSNorm weight: 1 + N(0, 0.05), as bf16 bits."""
    g = _gen(seed, device)
    return to_bits(1.0 + 0.05 * torch.randn(dim, generator=g, device=device, dtype=torch.float32))


def layer_matrices(shape: dict) -> list[tuple[str, int, int]]:
    """(name, N, K) of the linear layers of one decoder layer, each as stored
    (Wq, Wk, Wv, Wo, Wgate, Wup, Wdown)."""
    h, f = shape["hidden"], shape["ffn"]
    q = shape["n_q"] * shape["head_dim"]
    kv = shape["n_kv"] * shape["head_dim"]
    return [("wq", q, h), ("wk", kv, h), ("wv", kv, h), ("wo", h, q),
            ("wgate", f, h), ("wup", f, h), ("wdown", h, f)]
