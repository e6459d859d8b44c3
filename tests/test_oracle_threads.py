"""The oracle's item loops (logits rows, attention outputs, projection rows) give
bit-identical results on one host thread and on several: each item is computed
by one thread with the same loop body, so the thread count cannot change a bit."""
import math

import numpy as np

from entropy_gated_kv_decode_b300 import synth


def _with_threads(orc, n, fn):
    old = orc.get_threads()
    orc.set_threads(n)
    try:
        return fn()
    finally:
        orc.set_threads(old)


def test_row_stats_thread_count_invariant(orc):
    rng = np.random.default_rng(3)
    x = synth.make_logits(rng, 37, 4099, synth.BF16, 0.3)
    one = _with_threads(orc, 1, lambda: orc.row_stats(x))
    many = _with_threads(orc, 4, lambda: orc.row_stats(x))
    for a, b in zip(one, many):
        assert np.array_equal(a, b)


def test_attention_thread_count_invariant(orc):
    w = synth.scaled(synth.WORKLOADS["batched"], batch=2, seq_len=200, n_heads=6, n_kv_heads=2,
                     head_dim=64, qkv_std=1.0)
    a = synth.make_attention(np.random.default_rng(4), w, 20)
    cnt = np.array([20, 7], np.int32)
    scale = 1.0 / math.sqrt(w.head_dim)
    one = _with_threads(orc, 1, lambda: orc.attention(a.q, a.k_cache, a.v_cache, cnt, scale))
    many = _with_threads(orc, 3, lambda: orc.attention(a.q, a.k_cache, a.v_cache, cnt, scale))
    assert np.array_equal(np.isnan(one), np.isnan(many))
    assert np.array_equal(np.nan_to_num(one), np.nan_to_num(many))
    samples = np.array([[1, 6, 5], [0, 0, 0], [0, 19, 3]], np.int32)
    s1 = _with_threads(orc, 1, lambda: orc.attention(a.q, a.k_cache, a.v_cache, cnt, scale,
                                                     samples=samples))
    s3 = _with_threads(orc, 3, lambda: orc.attention(a.q, a.k_cache, a.v_cache, cnt, scale,
                                                     samples=samples))
    assert np.array_equal(s1, s3)
    assert np.array_equal(s1[0], one[1, 6, 5])


def test_projection_thread_count_invariant(orc):
    rng = np.random.default_rng(5)
    x = synth.f32_to_bf16_bits(rng.standard_normal((9, 64), dtype=np.float32))
    wt = synth.f32_to_bf16_bits(rng.standard_normal((48, 64), dtype=np.float32))
    one = _with_threads(orc, 1, lambda: orc.projection(x, wt))
    many = _with_threads(orc, 4, lambda: orc.projection(x, wt, rows=np.arange(9)))
    assert np.array_equal(one, many)
