"""Pins of the oracle's COVER dual-view attention.

"Stop the Flip-Flop" (COVER), Italian technical summary, "Metodologia: COVER",
item 1: seed positions (decoded tokens under verification) get [MASK] inputs; for
every other query the seed columns keep the K/V cached at the previous step (the
override); for a seed query the diagonal column is restored from the
masked-input K/V (leave-one-out, no self-leakage).  The checks: reduction to the
plain write-back + attention when nothing is a seed, exact cache contents,
leave-one-out and no-leak invariances, explicit per-query key matrices in numpy,
and the one-key closed form.
"""
import numpy as np
import pytest


def _case(rng, B=2, L=13, R=5, H=4, Hkv=2, d=8):
    q = rng.standard_normal((B, R, H, d))
    kn = rng.standard_normal((B, R, Hkv, d))
    vn = rng.standard_normal((B, R, Hkv, d))
    kc = rng.standard_normal((B, L, Hkv, d))
    vc = rng.standard_normal((B, L, Hkv, d))
    idx = np.stack([np.sort(rng.choice(L, R, replace=False)) for _ in range(B)]).astype(np.int32)
    cnt = np.full(B, R, np.int32)
    return q, kn, vn, kc, vc, idx, cnt


def test_no_seed_reduces_to_write_back_and_attention(orc):
    rng = np.random.default_rng(0)
    q, kn, vn, kc, vc, idx, cnt = _case(rng)
    cnt[1] = 3
    seed = np.zeros(idx.shape, np.uint8)
    k2, v2, out = orc.attention_cover(q, kn, vn, kc, vc, idx, cnt, seed, 0.4)
    k_ref, v_ref = orc.scatter_kv(kn, vn, idx, cnt, kc, vc)
    assert np.array_equal(k2, k_ref) and np.array_equal(v2, v_ref)
    want = orc.attention(q, k_ref, v_ref, cnt, 0.4)
    assert np.array_equal(np.isnan(out), np.isnan(want))
    assert np.allclose(out, want, rtol=1e-13, atol=1e-14, equal_nan=True)


def test_seed_positions_keep_the_previous_step_kv(orc):
    rng = np.random.default_rng(1)
    q, kn, vn, kc, vc, idx, cnt = _case(rng)
    seed = np.zeros(idx.shape, np.uint8)
    seed[0, [1, 3]] = 1
    seed[1, 0] = 1
    k2, v2, _ = orc.attention_cover(q, kn, vn, kc, vc, idx, cnt, seed, 0.4)
    for b in range(2):
        for r in range(cnt[b]):
            p = idx[b, r]
            want_k, want_v = (kc[b, p], vc[b, p]) if seed[b, r] else (kn[b, r], vn[b, r])
            assert np.array_equal(k2[b, p], want_k) and np.array_equal(v2[b, p], want_v)
        rest = np.setdiff1d(np.arange(kc.shape[1]), idx[b, :cnt[b]])
        assert np.array_equal(k2[b, rest], kc[b, rest]) and np.array_equal(v2[b, rest], vc[b, rest])


def test_leave_one_out_and_no_leak(orc):
    # A seed query never sees the token stored at its own position (the previous
    # step's K/V there), while every other query does; a seed's masked-input K/V
    # reach its own query only.
    rng = np.random.default_rng(2)
    q, kn, vn, kc, vc, idx, cnt = _case(rng, B=1, L=11, R=6)
    seed = np.zeros(idx.shape, np.uint8)
    seed[0, 2] = 1
    p = idx[0, 2]
    _, _, base = orc.attention_cover(q, kn, vn, kc, vc, idx, cnt, seed, 0.5)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[0, p] += 4.0
    vc2[0, p] -= 3.0
    _, _, moved = orc.attention_cover(q, kn, vn, kc2, vc2, idx, cnt, seed, 0.5)
    assert np.array_equal(moved[0, 2], base[0, 2])
    others = [r for r in range(6) if r != 2]
    assert all(not np.allclose(moved[0, r], base[0, r]) for r in others)
    kn2, vn2 = kn.copy(), vn.copy()
    kn2[0, 2] += 4.0
    vn2[0, 2] -= 3.0
    k3, v3, moved = orc.attention_cover(q, kn2, vn2, kc, vc, idx, cnt, seed, 0.5)
    assert not np.allclose(moved[0, 2], base[0, 2])
    assert np.array_equal(moved[0, others], base[0, others])
    assert np.array_equal(k3[0, p], kc[0, p]) and np.array_equal(v3[0, p], vc[0, p])


@pytest.mark.parametrize("H,Hkv", [(1, 1), (4, 2), (6, 1)])
def test_explicit_per_query_key_matrices(orc, H, Hkv):
    rng = np.random.default_rng(H)
    B, L, R, d = 2, 9, 4, 4
    q, kn, vn, kc, vc, idx, cnt = _case(rng, B, L, R, H, Hkv, d)
    seed = (rng.random(idx.shape) < 0.5).astype(np.uint8)
    _, _, out = orc.attention_cover(q, kn, vn, kc, vc, idx, cnt, seed, 0.7)
    for b in range(B):
        # the cache every query shares: non-seed rows written, seeds untouched
        K, V = kc[b].copy(), vc[b].copy()
        for r in range(R):
            if not seed[b, r]:
                K[idx[b, r]], V[idx[b, r]] = kn[b, r], vn[b, r]
        for r in range(R):
            Kr, Vr = K.copy(), V.copy()
            if seed[b, r]:  # its own column from the masked input
                Kr[idx[b, r]], Vr[idx[b, r]] = kn[b, r], vn[b, r]
            for h in range(H):
                g = h // (H // Hkv)
                s = Kr[:, g] @ q[b, r, h] * 0.7
                p = np.exp(s - s.max())
                p /= p.sum()
                assert np.allclose(out[b, r, h], p @ Vr[:, g], rtol=1e-12, atol=1e-13)


def test_single_key_seed_returns_its_masked_value(orc):
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 1, 2, 8))
    kn = rng.standard_normal((1, 1, 1, 8))
    vn = rng.standard_normal((1, 1, 1, 8))
    kc = rng.standard_normal((1, 1, 1, 8))
    vc = rng.standard_normal((1, 1, 1, 8))
    _, _, out = orc.attention_cover(q, kn, vn, kc, vc, np.zeros((1, 1), np.int32),
                                    np.ones(1, np.int32), np.ones((1, 1), np.uint8), 1.0)
    assert np.allclose(out[0, 0], np.broadcast_to(vn[0, 0, 0], (2, 8)), atol=1e-15)


def test_bad_index_is_rejected(orc):
    rng = np.random.default_rng(5)
    q, kn, vn, kc, vc, idx, cnt = _case(rng, B=1)
    idx[0, 0] = 99
    with pytest.raises(ValueError):
        orc.attention_cover(q, kn, vn, kc, vc, idx, cnt, np.zeros(idx.shape, np.uint8), 1.0)
