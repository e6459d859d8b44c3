"""Pins of the oracle's KV write-back and selective bidirectional attention.

EntropyCache, Italian summary, section 1: dLLM attention is bidirectional, every
position attends to all others; "Algoritmo di Funzionamento" step 2: the partial
forward recomputes K/V only for the selected tokens and reuses the cache for
the rest.  The checks use an explicitly materialised numpy softmax(Q K^T s) V,
closed-form special cases and invariances.
"""
import numpy as np
import pytest

from entropy_gated_kv_decode_b300 import synth


def _explicit(q, kc, vc, count, scale):
    """softmax(Q K^T * scale) V with whole matrices (numpy matmul), per (b, h)."""
    B, R, H, d = q.shape
    Hkv = kc.shape[2]
    out = np.full(q.shape, np.nan)
    for b in range(B):
        for h in range(H):
            g = h // (H // Hkv)
            Q = q[b, :count[b], h].astype(np.float64)
            K = kc[b, :, g].astype(np.float64)
            V = vc[b, :, g].astype(np.float64)
            S = Q @ K.T * scale
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            out[b, :count[b], h] = P @ V
    return out


@pytest.mark.parametrize("B,L,R,H,Hkv,d", [(1, 1, 1, 1, 1, 1), (1, 7, 3, 2, 2, 4),
                                           (2, 8, 5, 6, 2, 8), (3, 5, 5, 4, 1, 3)])
def test_attention_matches_explicit_matrices(orc, B, L, R, H, Hkv, d):
    rng = np.random.default_rng(B * 100 + L)
    q = rng.standard_normal((B, R, H, d))
    kc = rng.standard_normal((B, L, Hkv, d))
    vc = rng.standard_normal((B, L, Hkv, d))
    count = rng.integers(0, R + 1, size=B).astype(np.int32)
    count[0] = R
    scale = 1 / np.sqrt(d)
    got = orc.attention(q, kc, vc, count, scale)
    want = _explicit(q, kc, vc, count, scale)
    for b in range(B):
        assert np.allclose(got[b, :count[b]], want[b, :count[b]], rtol=1e-12, atol=1e-13)
        assert np.isnan(got[b, count[b]:]).all()


def test_identical_keys_give_the_mean_value(orc):
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 4, 2, 8))
    kc = np.broadcast_to(rng.standard_normal((1, 1, 2, 8)), (1, 9, 2, 8)).copy()
    vc = rng.standard_normal((1, 9, 2, 8))
    got = orc.attention(q, kc, vc, np.array([4], np.int32), 0.7)
    assert np.allclose(got[0], np.broadcast_to(vc[0].mean(axis=0), (4, 2, 8)), atol=1e-14)


def test_one_dominant_key_selects_its_value(orc):
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 1, 1, 16))
    kc = rng.standard_normal((1, 6, 1, 16)) * 0.01
    kc[0, 4, 0] = q[0, 0, 0] * 50.0
    vc = rng.standard_normal((1, 6, 1, 16))
    got = orc.attention(q, kc, vc, np.array([1], np.int32), 1.0)
    assert np.allclose(got[0, 0, 0], vc[0, 4, 0], atol=1e-12)


def test_key_permutation_invariance(orc):
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 3, 4, 8))
    kc = rng.standard_normal((1, 11, 2, 8))
    vc = rng.standard_normal((1, 11, 2, 8))
    perm = rng.permutation(11)
    a = orc.attention(q, kc, vc, np.array([3], np.int32), 0.35)
    b = orc.attention(q, kc[:, perm], vc[:, perm], np.array([3], np.int32), 0.35)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14, equal_nan=True)


def test_samples_agree_with_full_output(orc):
    rng = np.random.default_rng(4)
    q = rng.standard_normal((2, 5, 4, 8)).astype(np.float32)
    kc = rng.standard_normal((2, 13, 2, 8)).astype(np.float32)
    vc = rng.standard_normal((2, 13, 2, 8)).astype(np.float32)
    cnt = np.array([5, 3], np.int32)
    full = orc.attention(q, kc, vc, cnt, 0.5)
    samples = np.array([[0, 4, 3], [1, 2, 0], [1, 0, 1]])
    part = orc.attention(q, kc, vc, cnt, 0.5, samples=samples)
    for s, (b, r, h) in enumerate(samples):
        assert np.array_equal(part[s], full[b, r, h])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scatter_writes_exactly_the_selected_rows(orc, dtype):
    rng = np.random.default_rng(5)
    conv = (lambda x: x.astype(np.float32)) if dtype == "f32" else synth.f32_to_bf16_bits
    B, L, R, Hkv, d = 2, 20, 6, 3, 4
    kc = conv(rng.standard_normal((B, L, Hkv, d)))
    vc = conv(rng.standard_normal((B, L, Hkv, d)))
    kn = conv(rng.standard_normal((B, R, Hkv, d)))
    vn = conv(rng.standard_normal((B, R, Hkv, d)))
    cnt = np.array([6, 2], np.int32)
    idx = synth.random_index_set(rng, B, L, cnt, L)
    k2, v2 = orc.scatter_kv(kn, vn, idx, cnt, kc, vc)
    for b in range(B):
        sel = idx[b, :cnt[b]]
        assert np.array_equal(k2[b, sel], kn[b, :cnt[b]])
        assert np.array_equal(v2[b, sel], vn[b, :cnt[b]])
        rest = np.setdiff1d(np.arange(L), sel)
        assert np.array_equal(k2[b, rest], kc[b, rest])
        assert np.array_equal(v2[b, rest], vc[b, rest])


def test_bf16_inputs_widen_exactly(orc):
    rng = np.random.default_rng(6)
    q32 = rng.standard_normal((1, 2, 2, 8)).astype(np.float32)
    k32 = rng.standard_normal((1, 9, 1, 8)).astype(np.float32)
    v32 = rng.standard_normal((1, 9, 1, 8)).astype(np.float32)
    qb, kb, vb = (synth.f32_to_bf16_bits(x) for x in (q32, k32, v32))
    via_bits = orc.attention(qb, kb, vb, np.array([2], np.int32), 0.3)
    widened = [synth.bf16_bits_to_f32(x).astype(np.float64) for x in (qb, kb, vb)]
    via_f64 = orc.attention(*widened, np.array([2], np.int32), 0.3)
    assert np.array_equal(via_bits, via_f64)


@pytest.mark.parametrize("cuts", [[0, 5, 11], [0, 1, 2, 3, 17], [0, 9]])
def test_key_split_partials_combine_to_the_full_attention(orc, cuts):
    # The GPU path may cut a row's keys into pieces, keep per piece the raw-score
    # maximum m_s, l_s = sum 2^{(s - m_s) c} and the unnormalised O_s, and combine
    # out = sum_s 2^{(m_s - M) c} O_s / sum_s 2^{(m_s - M) c} l_s (M = max m_s, c =
    # scale * log2 e).  Pin that identity against the oracle's unsplit attention.
    rng = np.random.default_rng(len(cuts))
    L, R, H, d = 23, 4, 2, 8
    q = rng.standard_normal((1, R, H, d)) * 3
    kc = rng.standard_normal((1, L, H, d))
    vc = rng.standard_normal((1, L, H, d))
    count = np.array([R], np.int32)
    scale = 1 / np.sqrt(d)
    c = scale * np.log2(np.e)
    full = orc.attention(q, kc, vc, count, scale)
    bounds = cuts + [L]
    for r in range(R):
        for h in range(H):
            raw = kc[0, :, h] @ q[0, r, h]  # raw scores
            parts = []
            for a, z in zip(bounds[:-1], bounds[1:]):
                m = raw[a:z].max()
                p = np.exp2((raw[a:z] - m) * c)
                parts.append((m, p.sum(), p @ vc[0, a:z, h]))
            M = max(m for m, _, _ in parts)
            w = [np.exp2((m - M) * c) for m, _, _ in parts]
            out = sum(wi * o for wi, (_, _, o) in zip(w, parts)) / sum(wi * l for wi, (_, l, _) in zip(w, parts))
            assert np.allclose(out, full[0, r, h], rtol=1e-12, atol=1e-13)
