"""Float64 statements of the forward-pass operations between the matrix
products of one decode step of the evaluated models (Llama-3-8B, Qwen3-8B:
Cassandra paper, evaluation; Cassandra blog review, section 4).

TEST INFRASTRUCTURE ONLY (see the package docstring). Each function is the
plain definition, written out in numpy float64, with no blocking or fusion.
"""
from __future__ import annotations

import numpy as np


def _f64_of_bf16(bits) -> np.ndarray:
    b = np.asarray(bits).view(np.uint16) if np.asarray(bits).dtype != np.uint16 else np.asarray(bits)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rmsnorm(x, gamma_bits, eps: float) -> np.ndarray:
    """RMSNorm of each row: x / sqrt(mean(x^2) + eps) * gamma."""
    x = np.asarray(x, dtype=np.float64)
    g = _f64_of_bf16(gamma_bits)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope(x, positions, theta: float) -> np.ndarray:
    """Rotary embedding of heads of 128 values: in each head the pair
    (i, i + 64), i < 64, turns by the angle p * theta^(-i/64).
    x: [rows][H][128]; positions: [rows]."""
    x = np.asarray(x, dtype=np.float64)
    p = np.asarray(positions, dtype=np.float64)[:, None, None]
    i = np.arange(64, dtype=np.float64)[None, None, :]
    ang = p * theta ** (-i / 64.0)
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :64], x[..., 64:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def rope_split(qkv, n_q: int, n_kv: int, pos0: int, rows_per_seq: int, theta: float):
    """The fused QKV product split into q, k, v heads; q and k rotated at
    positions pos0 + row % rows_per_seq. Returns float64 (q, k, v)."""
    qkv = np.asarray(qkv, dtype=np.float64)
    rows = qkv.shape[0]
    h = qkv.reshape(rows, n_q + 2 * n_kv, 128)
    pos = pos0 + np.arange(rows) % rows_per_seq
    return rope(h[:, :n_q], pos, theta), rope(h[:, n_q:n_q + n_kv], pos, theta), h[:, n_q + n_kv:]


def silu_mul(gate_up) -> np.ndarray:
    """silu(gate) * up, silu(g) = g / (1 + exp(-g)); gate_up = [gate | up] per row."""
    gu = np.asarray(gate_up, dtype=np.float64)
    f = gu.shape[-1] // 2
    g, u = gu[..., :f], gu[..., f:]
    return g / (1.0 + np.exp(-g)) * u


def argmax(logits) -> np.ndarray:
    """Lowest index of the row maximum (NaN never wins)."""
    lg = np.asarray(logits, dtype=np.float64)
    lg = np.where(np.isnan(lg), -np.inf, lg)
    return np.argmax(lg, axis=-1)  # numpy returns the first occurrence


def embed(tokens, table_bits) -> np.ndarray:
    """Rows of the embedding table as float64."""
    return _f64_of_bf16(np.asarray(table_bits)[np.asarray(tokens)])
