"""Pins of the oracle's discrete decisions: confidence-ranked unmasking, the
max-entropy gate, the state update and the recompute index set.

EntropyCache, Italian summary, "Algoritmo di Funzionamento": step 1 decodes new
tokens and takes the maximum entropy E of their distributions; step 2 triggers
a full forward when E > tau and otherwise recomputes only the currently masked
tokens and the k most recently decoded ones.  The Arabic summary, "Algorithm
workflow" phase 3, keeps a log of decode times and picks the top k from it.
Each check below uses an independent formulation (Python sorting or rank
counting, exhaustive enumeration) rather than the oracle's own code.
"""
import itertools

import numpy as np
import pytest


def _state(batch, seq_len):
    return (np.ones((batch, seq_len), np.uint8), np.zeros((batch, seq_len), np.int32),
            np.full((batch, seq_len), -1, np.int32))


def test_unmask_hand_example(orc):
    # conf [0.9, 0.5, 0.9, 0.1] at positions [7, 3, 2, 5], n = 2 -> the rows at
    # positions 2 then 7 (equal confidence: lower position first)
    conf = np.array([0.9, 0.5, 0.9, 0.1])
    ent = np.array([0.3, 2.0, 0.4, 5.0])
    tok = np.array([11, 12, 13, 14], np.int32)
    im, tk, ds = _state(1, 8)
    res = orc.unmask_gate(conf, ent, tok, [0, 4], [7, 3, 2, 5], 8, 2, 0.35, 9, im, tk, ds)
    assert list(res["unmask_rows"][0]) == [2, 0]
    assert res["max_entropy"][0] == 0.4
    assert res["refresh"][0] == 1
    assert res["is_masked"][0, 2] == 0 and res["is_masked"][0, 7] == 0
    assert res["is_masked"][0, 3] == 1 and res["is_masked"][0, 5] == 1
    assert res["tokens"][0, 2] == 13 and res["tokens"][0, 7] == 11
    assert res["decode_step"][0, 2] == 9 and res["decode_step"][0, 7] == 9
    assert res["decode_step"][0, 3] == -1


def test_gate_is_strict(orc):
    # E == tau keeps the partial forward; the next float above tau refreshes.
    tau = np.float32(0.5)
    above = float(np.nextafter(np.float64(tau), 1.0))
    for e_val, expect in [(float(tau), 0), (above, 1), (0.25, 0)]:
        im, tk, ds = _state(1, 4)
        res = orc.unmask_gate([0.9], [e_val], [1], [0, 1], [0], 4, 1, tau, 0, im, tk, ds)
        assert res["refresh"][0] == expect


def test_gate_uses_only_the_unmasked_rows(orc):
    # the high-entropy row has low confidence and is not unmasked: no refresh
    im, tk, ds = _state(1, 4)
    res = orc.unmask_gate([0.9, 0.2], [0.1, 9.0], [1, 2], [0, 2], [0, 1], 4, 1, 1.0, 0,
                          im, tk, ds)
    assert list(res["unmask_rows"][0]) == [0]
    assert res["max_entropy"][0] == 0.1 and res["refresh"][0] == 0


def test_empty_sequence_and_short_sequence(orc):
    im, tk, ds = _state(2, 6)
    res = orc.unmask_gate([0.7, 0.8], [1.0, 3.0], [4, 5], [0, 0, 2], [1, 4], 6, 3, 2.0, 5,
                          im, tk, ds)
    assert list(res["unmask_rows"][0]) == [-1, -1, -1]
    assert res["max_entropy"][0] == -np.inf and res["refresh"][0] == 0
    assert list(res["unmask_rows"][1]) == [1, 0, -1]
    assert res["max_entropy"][1] == 3.0 and res["refresh"][1] == 1
    assert res["is_masked"][0].all()


def test_unmask_matches_python_sort_on_random_sequences(orc):
    rng = np.random.default_rng(21)
    for trial in range(200):
        batch = int(rng.integers(1, 5))
        seq_len = int(rng.integers(4, 40))
        counts = rng.integers(0, seq_len + 1, size=batch)
        off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        pos = np.concatenate([rng.choice(seq_len, size=c, replace=False) for c in counts]
                             ).astype(np.int32)
        n_rows = int(off[-1])
        # coarse confidences so that ties happen often
        conf = rng.integers(1, 6, size=n_rows) / 8.0
        ent = rng.uniform(0, 3, size=n_rows)
        tok = rng.integers(0, 100, size=n_rows).astype(np.int32)
        n = int(rng.integers(1, 6))
        tau = np.float32(rng.uniform(0, 3))
        im, tk, ds = _state(batch, seq_len)
        res = orc.unmask_gate(conf, ent, tok, off, pos, seq_len, n, tau, trial, im, tk, ds)
        for b in range(batch):
            rows = list(range(off[b], off[b + 1]))
            ranked = sorted(rows, key=lambda r: (-conf[r], pos[r]))[:n]
            got = [r for r in res["unmask_rows"][b] if r >= 0]
            assert got == ranked
            e = max((ent[r] for r in ranked), default=-np.inf)
            assert res["max_entropy"][b] == e
            assert res["refresh"][b] == int(e > float(tau))
            for r in ranked:
                assert res["is_masked"][b, pos[r]] == 0
                assert res["tokens"][b, pos[r]] == tok[r]
                assert res["decode_step"][b, pos[r]] == trial
            assert res["is_masked"][b].sum() == seq_len - len(ranked)


# ---------------------------------------------------------------------------
# recompute index set


def _by_rank_counting(is_masked, decode_step, lo, hi, k):
    """Independent formulation: position p is among the k most recent when fewer
    than k decoded positions q beat it (later step, or same step and lower position)."""
    L = len(is_masked)
    dec = [p for p in range(L) if decode_step[p] >= 0 and not is_masked[p]]
    chosen = set(p for p in range(lo, hi) if is_masked[p])
    for p in dec:
        better = sum(1 for q in dec if decode_step[q] > decode_step[p]
                     or (decode_step[q] == decode_step[p] and q < p))
        if better < k:
            chosen.add(p)
    return sorted(chosen)


def test_recompute_set_exhaustive_small_states(orc):
    L = 5
    cases = 0
    for masks in itertools.product([0, 1], repeat=L):
        for steps in itertools.product([-1, 0, 1], repeat=L):
            im = np.array([masks], np.uint8)
            ds = np.array([[s if not m else -1 for s, m in zip(steps, masks)]], np.int32)
            for lo, hi in [(0, L), (1, 4), (2, 2)]:
                for k in [0, 1, 2, 5]:
                    idx, cnt = orc.recompute_set(im, ds, np.zeros(1, np.uint8), lo, hi, k)
                    want = _by_rank_counting(im[0], ds[0], lo, hi, k)
                    assert list(idx[0, :cnt[0]]) == want
                    assert (idx[0, cnt[0]:] == -1).all()
                    cases += 1
    assert cases > 10000


def test_recompute_set_refresh_takes_everything(orc):
    im, _, ds = _state(3, 17)
    idx, cnt = orc.recompute_set(im, ds, np.array([1, 0, 1], np.uint8), 0, 4, 2)
    assert list(cnt) == [17, 4, 17]
    assert list(idx[0]) == list(range(17)) and list(idx[2]) == list(range(17))
    assert list(idx[1, :4]) == [0, 1, 2, 3]


def test_recompute_set_invariants_on_random_states(orc):
    rng = np.random.default_rng(4)
    for _ in range(50):
        B, L = int(rng.integers(1, 4)), int(rng.integers(8, 300))
        im = (rng.uniform(size=(B, L)) < 0.4).astype(np.uint8)
        ds = np.where(im == 1, -1, rng.integers(-1, 30, size=(B, L))).astype(np.int32)
        lo = int(rng.integers(0, L))
        hi = int(rng.integers(lo, L + 1))
        k = int(rng.integers(0, 40))
        idx, cnt = orc.recompute_set(im, ds, np.zeros(B, np.uint8), lo, hi, k)
        for b in range(B):
            sel = idx[b, :cnt[b]]
            assert np.all(np.diff(sel) > 0)  # ascending, hence disjoint
            n_masked = int(im[b, lo:hi].sum())
            n_dec = int(((ds[b] >= 0) & (im[b] == 0)).sum())
            assert cnt[b] == n_masked + min(k, n_dec)
            # every chosen decoded position is at least as recent as every unchosen one
            chosen = set(sel.tolist())
            dec_in = [ds[b, p] for p in chosen if ds[b, p] >= 0 and im[b, p] == 0]
            dec_out = [ds[b, p] for p in range(L) if p not in chosen and ds[b, p] >= 0
                       and im[b, p] == 0]
            if dec_in and dec_out:
                assert min(dec_in) >= max(dec_out)
