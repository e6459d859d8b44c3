"""float64 oracle of the pre-norm transformer layer the trajectory can run.

TEST INFRASTRUCTURE, like the rest of this package.

The pages evaluate EntropyCache on LLaDA-8B and Dream-7B (EntropyCache, Italian
summary, section 3) and describe no layer; their layers are pre-norm decoder
blocks with RMS normalisation, rotary position embeddings and a gated (SwiGLU)
MLP, which is the plain reading taken here:
    a = rms_norm(x, g1);  [q|k|v] = a W_qkv^T;  q, k = rope(q, k, positions)
    o = attention(q, K, V);  h = x + o W_o^T
    b = rms_norm(h, g2);  y = h + (silu(b W_gate^T) * (b W_up^T)) W_down^T
with rms_norm(x, g) = x / sqrt(mean(x^2) + eps) * g, silu(z) = z / (1 + e^-z),
and rope turning each pair (x_i, x_{i+d/2}) by p * theta^(-2i/d).  Every value is
widened to float64; nothing is rounded in between.
"""
from __future__ import annotations

import numpy as np

from entropy_gated_kv_decode_b300 import synth


def widen(a: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else \
        np.asarray(a, np.float64)


def rms_norm(x, g, eps):
    """x [..., n] -> x / sqrt(mean(x^2) + eps) * g."""
    x = widen(x)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * widen(g)


def rope(x, positions, theta):
    """x [r, heads, d] turned row by row: row j at positions[j]."""
    x = widen(x)
    d = x.shape[-1]
    half = d // 2
    freq = theta ** (-2.0 * np.arange(half) / d)
    ang = np.asarray(positions, np.float64)[:, None] * freq[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(z):
    return z / (1.0 + np.exp(-z))


def linear(x, w, mode=0, residual=None):
    """mode 0: x w^T; 1: residual + x w^T; 2: silu(x w_g^T) * (x w_u^T), w = [w_g; w_u]."""
    x, w = widen(x), widen(w)
    if mode == 2:
        f = w.shape[0] // 2
        return silu(x @ w[:f].T) * (x @ w[f:].T)
    y = x @ w.T
    return widen(residual) + y if mode == 1 else y
