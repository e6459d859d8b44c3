"""Pins of the oracle's pre-norm layer pieces (RMS norm, rotary embedding, the
linear layer's three forms).  The pages name the models (LLaDA-8B, Dream-7B) but
not their layers; the checks are the operations' defining properties: closed
forms, invariances, the relative-position property of rotary embeddings, and
library routines (numpy matmul, scipy's logistic function)."""
import numpy as np
import pytest
from scipy.special import expit

from oracle import layer


def test_rms_norm_closed_forms():
    rng = np.random.default_rng(0)
    g = rng.standard_normal(16)
    c = -2.5
    y = layer.rms_norm(np.full((3, 16), c), g, 0.0)
    assert np.allclose(y, np.sign(c) * g, atol=1e-15)  # a constant row keeps only its sign
    eps = 0.3
    y = layer.rms_norm(np.full((1, 16), c), g, eps)
    assert np.allclose(y, c / np.sqrt(c * c + eps) * g, atol=1e-15)
    x = rng.standard_normal((5, 16))
    y = layer.rms_norm(x, np.ones(16), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0)  # unit RMS
    assert np.allclose(layer.rms_norm(7.0 * x, g, 0.0), layer.rms_norm(x, g, 0.0))


def test_rope_identity_norms_and_composition():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((4, 3, 16))
    theta = 10000.0
    assert np.allclose(layer.rope(x, [0, 0, 0, 0], theta), x, atol=1e-15)
    y = layer.rope(x, [1, 5, 100, 8191], theta)
    pair = lambda a: a[..., :8] ** 2 + a[..., 8:] ** 2  # noqa: E731
    assert np.allclose(pair(y), pair(x))  # every pair keeps its length
    two = layer.rope(layer.rope(x, [3, 4, 5, 6], theta), [10, 20, 30, 40], theta)
    assert np.allclose(two, layer.rope(x, [13, 24, 35, 46], theta))


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 1, 32))
    k = rng.standard_normal((1, 1, 32))
    theta = 500000.0
    s = [float(np.sum(layer.rope(q, [m + 7], theta) * layer.rope(k, [m], theta)))
         for m in (0, 3, 100, 4000)]
    assert np.allclose(s, s[0])
    assert not np.isclose(s[0], float(np.sum(layer.rope(q, [9], theta) * layer.rope(k, [0], theta))))


def test_rope_matches_complex_rotation():
    # the pairs (x_i, x_{i+d/2}) as complex numbers multiplied by e^{i p w_i}
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 1, 8))
    pos = np.array([3, 11])
    w = 10000.0 ** (-np.arange(4) * 2 / 8)
    z = (x[..., :4] + 1j * x[..., 4:]) * np.exp(1j * pos[:, None, None] * w)
    assert np.allclose(layer.rope(x, pos, 10000.0), np.concatenate([z.real, z.imag], axis=-1))


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_linear_forms(mode):
    rng = np.random.default_rng(4 + mode)
    x = rng.standard_normal((5, 8))
    w = rng.standard_normal((12, 8))
    res = rng.standard_normal((5, 6 if mode == 2 else 12))
    y = layer.linear(x, w, mode, res)
    if mode == 0:
        assert np.allclose(y, np.matmul(x, w.T))
    elif mode == 1:
        assert np.allclose(y, res + np.matmul(x, w.T))
    else:
        g, u = np.matmul(x, w[:6].T), np.matmul(x, w[6:].T)
        assert np.allclose(y, g * expit(g) * u)  # silu(z) = z * logistic(z)
        assert np.allclose(layer.linear(x, np.concatenate([w[:6], 0 * w[6:]]), 2), 0.0)
