"""Pins of the oracle's COVER seed score.

"Stop the Flip-Flop" (COVER), Italian technical summary, "Metodologia: COVER",
item 2: a decoded token is scored by u (1 + d_in) / (1 + d_out), u its entropy,
d_in how much the still-masked positions attend to it, d_out how much it attends
to the positions drafted at this step; the seeds are the highest scores.  The
readings (head-averaged attention probabilities of one layer, summed over the
masked queries for d_in and over the drafted keys for d_out) are pinned by
closed forms: uniform attention, attention concentrated on one key per query
(counts, which tell d_in from d_out and each head's key-value head from
another's), two keys (the logistic function), and the ranking rule.
"""
import numpy as np
import pytest
from scipy.special import expit

from entropy_gated_kv_decode_b300 import synth


def _layout(rng, B, L, R):
    idx = np.stack([np.sort(rng.choice(L, R, replace=False)) for _ in range(B)]).astype(np.int32)
    return idx, np.full(B, R, np.int32)


def test_uniform_attention_closed_form(orc):
    # q = 0: every probability is 1/L, so d_in = (#masked queries) / L and
    # d_out = (#drafted keys) / L for every candidate
    rng = np.random.default_rng(0)
    B, L, R, H, Hkv, d = 2, 40, 9, 4, 2, 8
    q = np.zeros((B, R, H, d))
    kc = rng.standard_normal((B, L, Hkv, d))
    idx, cnt = _layout(rng, B, L, R)
    role = rng.integers(0, 4, (B, R)).astype(np.uint8)
    role[:, 0], role[:, 1] = 1, 2
    drafted = (rng.random((B, L)) < 0.2).astype(np.uint8)
    u = rng.random((B, R)) * 3
    d_in, d_out, score, _ = orc.cover_seed_score(q, kc, idx, cnt, role, drafted, u, 0.3, 2)
    for b in range(B):
        n_masked = np.count_nonzero(role[b] & 1)
        n_drafted = np.count_nonzero(drafted[b])
        cand = (role[b] & 2) != 0
        assert np.allclose(d_in[b, cand], n_masked / L, rtol=1e-13)
        assert np.allclose(d_out[b, cand], n_drafted / L, rtol=1e-13)
        want = u[b, cand] * (1 + n_masked / L) / (1 + n_drafted / L)
        assert np.allclose(score[b, cand], want, rtol=1e-13)
        assert np.isnan(score[b, ~cand]).all() and np.isnan(d_in[b, ~cand]).all()


def test_concentrated_attention_counts(orc):
    # Every key is a scaled basis vector (a different permutation per key-value
    # head) and every query points at one key with a score of 80 against 0 for
    # the rest, so a^h_{r,j} is 1 at its target and 0 (1e-35) elsewhere:
    # d_in(c) = (1/H) #{(h, masked r): target_h(r) = p_c},
    # d_out(c) = (1/H) #{h: target_h(c) drafted}.
    rng = np.random.default_rng(1)
    B, L, R, H, Hkv, d = 2, 12, 8, 6, 2, 16
    G = H // Hkv
    perm = [rng.permutation(d)[:L] for _ in range(Hkv)]
    kc = np.zeros((B, L, Hkv, d))
    for g in range(Hkv):
        kc[:, np.arange(L), g, perm[g]] = 4.0
    idx, cnt = _layout(rng, B, L, R)
    target = rng.integers(0, L, (B, R, H))
    for b in range(B):  # make some masked queries aim at candidate positions
        target[b, 0, :] = idx[b, 5]
        target[b, 1, ::2] = idx[b, 6]
    q = np.zeros((B, R, H, d))
    for b in range(B):
        for r in range(R):
            for h in range(H):
                q[b, r, h, perm[h // G][target[b, r, h]]] = 5.0
    scale = 4.0  # 4 * 5 * 4 = 80
    role = np.zeros((B, R), np.uint8)
    role[:, :4] = 1
    role[:, 3] |= 2  # a row may be both
    role[:, 5:] = 2
    drafted = np.zeros((B, L), np.uint8)
    drafted[:, ::3] = 1
    u = np.ones((B, R))
    d_in, d_out, score, _ = orc.cover_seed_score(q, kc, idx, cnt, role, drafted, u, scale, 3)
    for b in range(B):
        for c in range(R):
            if not role[b, c] & 2:
                assert np.isnan(d_in[b, c])
                continue
            hits = sum(1 for h in range(H) for r in range(R)
                       if role[b, r] & 1 and target[b, r, h] == idx[b, c])
            outs = sum(1 for h in range(H) if drafted[b, target[b, c, h]])
            assert d_in[b, c] == pytest.approx(hits / H, abs=1e-12)
            assert d_out[b, c] == pytest.approx(outs / H, abs=1e-12)
            assert score[b, c] == pytest.approx((1 + hits / H) / (1 + outs / H), abs=1e-12)
        assert d_in[b, 5] >= 1.0 and d_in[b, 6] >= 0.5


def test_two_keys_logistic(orc):
    # L = 2: a row's weight on key 0 is expit(scale * (s_0 - s_1))
    rng = np.random.default_rng(2)
    d = 8
    kc = rng.standard_normal((1, 2, 1, d))
    q = rng.standard_normal((1, 2, 1, d))
    idx = np.array([[0, 1]], np.int32)
    cnt = np.array([2], np.int32)
    role = np.array([[1, 2]], np.uint8)     # row 0 (position 0) masked, row 1 (position 1) candidate
    drafted = np.array([[1, 0]], np.uint8)  # position 0 drafted at this step
    scale = 0.7
    d_in, d_out, score, seeds = orc.cover_seed_score(q, kc, idx, cnt, role, drafted,
                                                     np.array([[0.0, 1.5]]), scale, 2)
    s = scale * np.einsum("rd,jd->rj", q[0, :, 0], kc[0, :, 0])
    a_masked_on_1 = expit(s[0, 1] - s[0, 0])
    a_cand_on_0 = expit(s[1, 0] - s[1, 1])
    assert d_in[0, 1] == pytest.approx(a_masked_on_1, rel=1e-14)
    assert d_out[0, 1] == pytest.approx(a_cand_on_0, rel=1e-14)
    assert score[0, 1] == pytest.approx(1.5 * (1 + a_masked_on_1) / (1 + a_cand_on_0), rel=1e-14)
    assert seeds.tolist() == [[1, -1]]


def test_ranking_ties_padding_and_nan(orc):
    # uniform attention: every candidate has the same d_in and d_out, so the
    # score orders as u; equal scores go to the lower position, a NaN score last
    rng = np.random.default_rng(3)
    B, L, R, H, d = 1, 30, 7, 2, 4
    q = np.zeros((B, R, H, d))
    kc = rng.standard_normal((B, L, H, d))
    idx = np.array([[2, 4, 9, 11, 17, 20, 28]], np.int32)
    cnt = np.array([R], np.int32)
    role = np.array([[2, 2, 1, 2, 2, 0, 2]], np.uint8)
    u = np.array([[1.0, 5.0, 9.0, 5.0, np.nan, 7.0, 2.0]])
    drafted = np.zeros((B, L), np.uint8)
    _, _, score, seeds = orc.cover_seed_score(q, kc, idx, cnt, role, drafted, u, 1.0, 7)
    # candidates: pos 2 (u 1), 4 (5), 11 (5), 17 (NaN), 28 (2); rows 9 and 20 are not
    assert seeds.tolist() == [[4, 11, 28, 2, 17, -1, -1]]
    _, _, _, top2 = orc.cover_seed_score(q, kc, idx, cnt, role, drafted, u, 1.0, 2)
    assert top2.tolist() == [[4, 11]]
    _, _, _, none = orc.cover_seed_score(q, kc, idx, cnt, role, drafted, u, 1.0, 0)
    assert none.shape == (1, 0)


def test_rows_outside_the_roles_or_past_count_do_not_count(orc):
    rng = np.random.default_rng(4)
    B, L, R, H, Hkv, d = 2, 25, 10, 4, 4, 8
    q = rng.standard_normal((B, R, H, d))
    kc = rng.standard_normal((B, L, Hkv, d))
    idx, cnt = _layout(rng, B, L, R)
    cnt[1] = 6
    role = np.array([[1, 2, 0, 3, 1, 2, 0, 2, 1, 0]] * 2, np.uint8)
    drafted = (rng.random((B, L)) < 0.3).astype(np.uint8)
    u = rng.random((B, R))
    base = orc.cover_seed_score(q, kc, idx, cnt, role, drafted, u, 0.5, 4)
    q2, role2, u2 = q.copy(), role.copy(), u.copy()
    q2[:, [2, 6, 9]] = rng.standard_normal((B, 3, H, d))  # role-0 rows
    q2[1, 6:] = rng.standard_normal((R - 6, H, d))        # rows past count
    role2[1, 6:] = 3
    u2[1, 6:] = 100.0
    moved = orc.cover_seed_score(q2, kc, idx, cnt, role2, drafted, u2, 0.5, 4)
    for x, y in zip(base, moved):
        assert np.array_equal(x, y, equal_nan=True)
    # the keys do count, at every position
    kc2 = kc.copy()
    kc2[0, int(np.flatnonzero(drafted[0])[0])] += 1.0
    assert not np.allclose(orc.cover_seed_score(q, kc2, idx, cnt, role, drafted, u, 0.5, 4)[1][0],
                           base[1][0], equal_nan=True)


def test_score_is_linear_in_u(orc):
    rng = np.random.default_rng(5)
    B, L, R, H, d = 1, 20, 6, 2, 8
    q = rng.standard_normal((B, R, H, d))
    kc = rng.standard_normal((B, L, H, d))
    idx, cnt = _layout(rng, B, L, R)
    role = np.array([[1, 1, 2, 2, 3, 2]], np.uint8)
    drafted = (rng.random((B, L)) < 0.3).astype(np.uint8)
    u = rng.random((B, R)) + 0.5
    d_in, d_out, s1, _ = orc.cover_seed_score(q, kc, idx, cnt, role, drafted, u, 0.4, 2)
    d_in2, d_out2, s2, _ = orc.cover_seed_score(q, kc, idx, cnt, role, drafted, 2.5 * u, 0.4, 2)
    assert np.array_equal(d_in, d_in2, equal_nan=True) and np.array_equal(d_out, d_out2, equal_nan=True)
    c = (role[0] & 2) != 0
    assert np.allclose(s2[0, c], 2.5 * s1[0, c], rtol=1e-15)
    _, _, s0, _ = orc.cover_seed_score(q, kc, idx, cnt, role, drafted, 0 * u, 0.4, 2)
    assert np.all(s0[0, c] == 0.0)


def test_bf16_inputs_read_as_their_exact_values(orc):
    rng = np.random.default_rng(6)
    B, L, R, H, Hkv, d = 2, 33, 7, 4, 2, 16
    q = synth.f32_to_bf16_bits(rng.standard_normal((B, R, H, d), dtype=np.float32))
    kc = synth.f32_to_bf16_bits(rng.standard_normal((B, L, Hkv, d), dtype=np.float32))
    idx, cnt = _layout(rng, B, L, R)
    role = rng.integers(0, 4, (B, R)).astype(np.uint8)
    drafted = (rng.random((B, L)) < 0.25).astype(np.uint8)
    u = rng.random((B, R))
    wide = lambda a: synth.bf16_bits_to_f32(a).astype(np.float64)  # noqa: E731
    got = orc.cover_seed_score(q, kc, idx, cnt, role, drafted, u, 0.25, 3)
    want = orc.cover_seed_score(wide(q), wide(kc), idx, cnt, role, drafted, u, 0.25, 3)
    for x, y in zip(got, want):
        assert np.array_equal(x, y, equal_nan=True)


def test_bad_arguments_are_rejected(orc):
    rng = np.random.default_rng(7)
    q = np.zeros((1, 3, 2, 4))
    kc = np.zeros((1, 5, 2, 4))
    role = np.full((1, 3), 3, np.uint8)
    drafted = np.zeros((1, 5), np.uint8)
    u = rng.random((1, 3))
    with pytest.raises(ValueError):
        orc.cover_seed_score(q, kc, np.array([[0, 1, 5]], np.int32), np.array([3], np.int32), role,
                             drafted, u, 1.0, 1)
    with pytest.raises(ValueError):
        orc.cover_seed_score(q, kc, np.array([[0, 1, 2]], np.int32), np.array([4], np.int32), role,
                             drafted, u, 1.0, 1)
