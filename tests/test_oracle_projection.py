"""Pins of the oracle's first-layer input gather and Q/K/V projection.

EntropyCache, Italian summary, "Algoritmo di Funzionamento" step 2: the partial
forward recomputes the queries, keys and values of the selected tokens only;
section 1: a position holds [MASK] until its token is decoded.  The projection
is pinned against numpy's float64 matmul (an independent library routine), an
identity weight and exactly representable integer products; the gather against
plain fancy indexing.
"""
import numpy as np

from entropy_gated_kv_decode_b300 import synth


def test_projection_matches_numpy_matmul(orc):
    rng = np.random.default_rng(0)
    x = rng.standard_normal((9, 40))
    w = rng.standard_normal((15, 40))
    assert np.allclose(orc.projection(x, w), x @ w.T, rtol=1e-13, atol=1e-13)
    rows = np.array([8, 0, 3])
    assert np.allclose(orc.projection(x, w, rows=rows), (x @ w.T)[rows], rtol=1e-13, atol=1e-13)


def test_projection_identity_and_exact_integers(orc):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((4, 16)).astype(np.float32)
    assert np.array_equal(orc.projection(x, np.eye(16, dtype=np.float32)), x.astype(np.float64))
    # small integers are exact in bf16 and their products sum exactly in float64
    xi = rng.integers(-8, 9, size=(6, 64)).astype(np.float32)
    wi = rng.integers(-8, 9, size=(12, 64)).astype(np.float32)
    got = orc.projection(synth.f32_to_bf16_bits(xi), synth.f32_to_bf16_bits(wi))
    want = xi.astype(np.int64) @ wi.astype(np.int64).T
    assert np.array_equal(got, want.astype(np.float64))


def test_embed_rows_is_a_row_gather(orc):
    rng = np.random.default_rng(2)
    V, hidden, B, L = 50, 8, 2, 12
    table = synth.f32_to_bf16_bits(rng.standard_normal((V + 1, hidden)).astype(np.float32))
    tokens = rng.integers(0, V, size=(B, L)).astype(np.int32)
    is_masked = (rng.uniform(size=(B, L)) < 0.5).astype(np.uint8)
    cnt = np.array([5, 3], np.int32)
    idx = synth.random_index_set(rng, B, L, cnt, stride=7)
    x = orc.embed_rows(table, idx, cnt, tokens, is_masked, V, r_max=6)
    for b in range(B):
        for r in range(cnt[b]):
            p = idx[b, r]
            want = table[V] if is_masked[b, p] else table[tokens[b, p]]
            assert np.array_equal(x[b, r], want)
        assert not x[b, cnt[b]:].any()
