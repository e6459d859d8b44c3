"""Pins of the oracle's attention under SimSD's temporal causal mask.

SimSD, Italian technical summary, "Metodologia: SimSD": item 1 lays the input
out as prompt + data section D + mask section (each response position k has a
data token D_k and a prediction slot); item 2 lets a mask slot attend to data
tokens of earlier steps (tau(j) < tau(i)) and to mask slots of the same or
later steps (tau(j) >= tau(i)).  The checks use a visibility table worked by
hand (tests/golden/simsd_visibility.txt), an explicit numpy masked softmax,
reductions to the plain attention over a subset of the keys, and the counting
properties a permutation step map implies.
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "simsd_visibility.txt")


def _golden():
    section = tau = None
    vis = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        if line.startswith("section"):
            section = np.array(line.split()[1:], np.uint8)
        elif line.startswith("tau"):
            tau = np.array(line.split()[1:], np.int32)
        else:
            head, rest = line.split(":")
            vis[int(head.split()[1])] = [int(x) for x in rest.split()]
    return section, tau, vis


def _layout(rng, batch, prompt, blk):
    """Sections and step labels of `batch` sequences: prompt, data, mask; one step
    map (a permutation of 1..blk) per sequence shared by each data/mask pair."""
    L = prompt + 2 * blk
    section = np.zeros((batch, L), np.uint8)
    tau = np.zeros((batch, L), np.int32)
    for b in range(batch):
        mu = rng.permutation(blk) + 1
        section[b, prompt:prompt + blk] = 1
        section[b, prompt + blk:] = 2
        tau[b, prompt:prompt + blk] = mu
        tau[b, prompt + blk:] = mu
    return section, tau


def _visible_sets(orc, section, tau):
    """Visibility of every query of one sequence, read off the oracle: q = 0 gives
    uniform weights over the visible keys, V = identity turns the output row into
    that set's indicator divided by its size."""
    L = section.shape[0]
    q = np.zeros((1, L, 1, L))
    kc = np.random.default_rng(0).standard_normal((1, L, 1, L))
    vc = np.eye(L).reshape(1, L, 1, L)
    idx = np.arange(L, dtype=np.int32)[None]
    out = orc.attention_simsd(q, kc, vc, idx, np.array([L], np.int32), section[None], tau[None], 1.0)
    sets = []
    for i in range(L):
        row = out[0, i, 0]
        nz = np.flatnonzero(row > 0)
        assert np.allclose(row[nz], 1.0 / len(nz), rtol=0, atol=1e-15)
        assert np.all(row[row <= 0] == 0)
        sets.append(set(nz.tolist()))
    return sets


def test_hand_worked_visibility(orc):
    section, tau, vis = _golden()
    sets = _visible_sets(orc, section, tau)
    for i, want in vis.items():
        assert sets[i] == set(want), f"query {i}"


@pytest.mark.parametrize("H,Hkv,d", [(1, 1, 4), (4, 2, 8), (6, 1, 3)])
def test_golden_layout_matches_explicit_masked_softmax(orc, H, Hkv, d):
    section, tau, vis = _golden()
    L = len(section)
    rng = np.random.default_rng(H * 10 + d)
    q = rng.standard_normal((1, L, H, d)) * 2
    kc = rng.standard_normal((1, L, Hkv, d))
    vc = rng.standard_normal((1, L, Hkv, d))
    perm = rng.permutation(L).astype(np.int32)  # query rows in any order
    scale = 0.6
    got = orc.attention_simsd(q, kc, vc, perm[None], np.array([L], np.int32), section[None],
                              tau[None], scale)
    mask = np.zeros((L, L), bool)
    for i, keys in vis.items():
        mask[i, keys] = True
    for h in range(H):
        g = h // (H // Hkv)
        S = q[0, :, h] @ kc[0, :, g].T * scale
        S = np.where(mask[perm], S, -np.inf)
        P = np.exp(S - S.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        assert np.allclose(got[0, :, h], P @ vc[0, :, g], rtol=1e-12, atol=1e-13)


def test_prompt_only_reduces_to_plain_attention(orc):
    rng = np.random.default_rng(7)
    B, L, R, H, Hkv, d = 2, 11, 4, 4, 2, 8
    q = rng.standard_normal((B, R, H, d))
    kc = rng.standard_normal((B, L, Hkv, d))
    vc = rng.standard_normal((B, L, Hkv, d))
    cnt = np.array([4, 2], np.int32)
    idx = np.stack([rng.choice(L, R, replace=False) for _ in range(B)]).astype(np.int32)
    z8 = np.zeros((B, L), np.uint8)
    got = orc.attention_simsd(q, kc, vc, idx, cnt, z8, np.zeros((B, L), np.int32), 0.4)
    want = orc.attention(q, kc, vc, cnt, 0.4)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.allclose(got, want, rtol=1e-13, atol=1e-14, equal_nan=True)


def test_first_and_last_steps_reduce_to_attention_over_a_key_subset(orc):
    # The slot decoded first sees no data token and the whole mask section; the
    # slot decoded last sees every other data token and only itself among the
    # slots; the data token of the last step sees the whole data section.
    rng = np.random.default_rng(8)
    P0, blk, H, Hkv, d = 6, 5, 4, 2, 8
    section, tau = _layout(rng, 1, P0, blk)
    L = P0 + 2 * blk
    q = rng.standard_normal((1, L, H, d))
    kc = rng.standard_normal((1, L, Hkv, d))
    vc = rng.standard_normal((1, L, Hkv, d))
    idx = np.arange(L, dtype=np.int32)[None]
    got = orc.attention_simsd(q, kc, vc, idx, np.array([L], np.int32), section, tau, 0.5)
    prompt = list(range(P0))
    data = list(range(P0, P0 + blk))
    slots = list(range(P0 + blk, L))
    first = slots[int(np.argmax(tau[0, slots] == 1))]
    last = slots[int(np.argmax(tau[0, slots] == blk))]
    last_data = data[int(np.argmax(tau[0, data] == blk))]
    cases = [(first, prompt + slots),
             (last, prompt + [j for j in data if tau[0, j] < blk] + [last]),
             (last_data, prompt + data)]
    for i, keys in cases:
        keys = np.array(sorted(keys))
        sub = orc.attention(q[:, i:i + 1], kc[:, keys], vc[:, keys], np.array([1], np.int32), 0.5)
        assert np.allclose(got[0, i], sub[0, 0], rtol=1e-13, atol=1e-14)


def test_a_slot_never_sees_its_own_reference_token(orc):
    # Item 2's point: the data token of the slot's own step is not yet revealed.
    rng = np.random.default_rng(9)
    P0, blk, H, d = 3, 4, 2, 4
    section, tau = _layout(rng, 1, P0, blk)
    L = P0 + 2 * blk
    q = rng.standard_normal((1, L, H, d))
    kc = rng.standard_normal((1, L, H, d))
    vc = rng.standard_normal((1, L, H, d))
    idx = np.arange(L, dtype=np.int32)[None]
    cnt = np.array([L], np.int32)
    base = orc.attention_simsd(q, kc, vc, idx, cnt, section, tau, 0.5)
    for k in range(blk):
        slot, ref = P0 + blk + k, P0 + k
        k2, v2 = kc.copy(), vc.copy()
        k2[0, ref] += 5.0
        v2[0, ref] -= 3.0
        moved = orc.attention_simsd(q, k2, v2, idx, cnt, section, tau, 0.5)
        assert np.array_equal(moved[0, slot], base[0, slot])
        k3 = kc.copy()
        k3[0, slot] += 5.0  # the slot itself is always visible
        moved = orc.attention_simsd(q, k3, vc, idx, cnt, section, tau, 0.5)
        assert not np.allclose(moved[0, slot], base[0, slot])


@pytest.mark.parametrize("seed", range(4))
def test_visible_set_sizes_follow_the_step_order(orc, seed):
    rng = np.random.default_rng(seed)
    P0, blk = int(rng.integers(0, 5)), int(rng.integers(1, 7))
    section, tau = _layout(rng, 1, P0, blk)
    sets = _visible_sets(orc, section[0], tau[0])
    prompt = set(range(P0))
    data = set(range(P0, P0 + blk))
    slots = set(range(P0 + blk, P0 + 2 * blk))
    by_step = sorted(slots, key=lambda i: tau[0, i])
    prev_d, prev_m = set(), set(slots)
    for s, i in enumerate(by_step, start=1):
        assert prompt <= sets[i]
        d_vis, m_vis = sets[i] & data, sets[i] & slots
        assert len(d_vis) == s - 1 and len(m_vis) == blk - s + 1
        assert prev_d <= d_vis and m_vis <= prev_m  # data grows, slots shrink
        prev_d, prev_m = d_vis, m_vis
    for i in data:
        assert sets[i] & slots == set() and prompt <= sets[i]
        assert len(sets[i] & data) == tau[0, i]
    for i in prompt:
        assert sets[i] == prompt


def test_samples_agree_with_full_output(orc):
    rng = np.random.default_rng(10)
    section, tau = _layout(rng, 2, 4, 3)
    B, L, H, Hkv, d = 2, 10, 4, 2, 8
    q = rng.standard_normal((B, 6, H, d)).astype(np.float32)
    kc = rng.standard_normal((B, L, Hkv, d)).astype(np.float32)
    vc = rng.standard_normal((B, L, Hkv, d)).astype(np.float32)
    idx = np.tile(np.arange(4, 10, dtype=np.int32), (B, 1))
    cnt = np.array([6, 5], np.int32)
    full = orc.attention_simsd(q, kc, vc, idx, cnt, section, tau, 0.3)
    samples = np.array([[0, 5, 3], [1, 4, 0], [1, 0, 1]])
    part = orc.attention_simsd(q, kc, vc, idx, cnt, section, tau, 0.3, samples=samples)
    for s, (b, r, h) in enumerate(samples):
        assert np.array_equal(part[s], full[b, r, h])
    assert np.isnan(full[1, 5]).all()


def test_bad_layouts_are_rejected(orc):
    rng = np.random.default_rng(11)
    section, tau = _layout(rng, 1, 2, 2)
    L = 6
    q = np.zeros((1, 2, 1, 4))
    kc = np.zeros((1, L, 1, 4))
    idx = np.array([[4, 5]], np.int32)
    cnt = np.array([2], np.int32)
    bad_sec = section.copy()
    bad_sec[0, 1] = 3
    bad_tau = tau.copy()
    bad_tau[0, 3] = 0
    for sec, tl, ix in [(bad_sec, tau, idx), (section, bad_tau, idx),
                        (section, tau, np.array([[4, 6]], np.int32))]:
        with pytest.raises(ValueError):
            orc.attention_simsd(q, kc, kc, ix, cnt, sec, tl, 1.0)
