"""Pins of the oracle's whole-trajectory composition.

EntropyCache, Italian summary, "Algoritmo di Funzionamento": step 0 is a full
forward; each step decodes, gates on E > tau, and the next forward recomputes
either everything or the masked tokens of the active block plus the k most
recently decoded ones.  Checked here: the schedule's invariants, the two
degenerate thresholds (never / always refresh), and, for an always-refresh
trajectory, the layers' numerics against a dense numpy forward written from
whole matrices (every row recomputed, so no cache state carries over)."""
import math

import numpy as np

import oracle.trajectory as otraj
from entropy_gated_kv_decode_b300 import synth

W = synth.scaled(synth.WORKLOADS["trajectory"], vocab=500, seq_len=96, prompt_len=64, block=8,
                 n_heads=2, n_kv_heads=2, head_dim=4, n_layers=2, n_steps=16)


def test_schedule_invariants():
    recs, final = otraj.run(W, 1)
    L, k = W.seq_len, W.k
    assert recs[0]["full"] and recs[0]["rows"] == L
    decoded = 0
    for t, r in enumerate(recs):
        lo, hi = synth.trajectory_block(W, t)
        assert np.all((r["row_pos"] >= lo) & (r["row_pos"] < hi))
        assert len(r["row_pos"]) == synth.trajectory_rows_per_step(W)[t]
        sel = [u for u in r["unmask_rows"] if u >= 0]
        assert len(sel) == min(W.n_unmask, len(r["row_pos"]))
        e = max(r["entropy"][u] for u in sel)
        assert r["max_entropy"] == e and r["refresh"] == int(e > float(np.float32(W.tau)))
        if t > 0:
            assert r["full"] == bool(recs[t - 1]["refresh"])
            if not r["full"]:
                masked = len(r["row_pos"])
                assert r["rows"] == masked + min(k, decoded)
        decoded += len(sel)
    assert final["is_masked"].sum() == 0
    assert (final["decode_step"][0, W.prompt_len:] >= 0).all()


def test_degenerate_thresholds():
    never = synth.scaled(W, tau=1e9)
    recs, _ = otraj.run(never, 2)
    assert [r["full"] for r in recs] == [True] + [False] * (len(recs) - 1)
    always = synth.scaled(W, tau=-1.0)
    recs, _ = otraj.run(always, 2)
    assert all(r["full"] for r in recs) and all(r["rows"] == W.seq_len for r in recs)


def test_always_refresh_forward_matches_dense_numpy():
    w = synth.scaled(W, tau=-1.0, n_steps=3)
    recs, final = otraj.run(w, 4, layers=2)
    H, d = w.n_heads, w.head_dim
    hid = H * d
    table = synth.bf16_bits_to_f32(synth.trajectory_embedding(4, w.vocab, hid)).astype(np.float64)
    tokens = final["tokens"][0].copy()
    # state before the last step's decode: undo the last step's unmasking
    im = final["is_masked"][0].copy()
    last = recs[-1]
    for u in last["unmask_rows"]:
        if u >= 0:
            im[last["row_pos"][u]] = 1
    x = np.where(im[:, None] == 1, table[w.vocab], table[np.where(im == 1, 0, tokens)])
    for layer in range(2):
        wq = synth.bf16_bits_to_f32(synth.trajectory_weights(4, layer, hid, hid)).astype(np.float64)
        q, k, v = (x @ wq[i * hid:(i + 1) * hid].T for i in range(3))
        outs = []
        for h in range(H):
            s = q[:, h * d:(h + 1) * d] @ k[:, h * d:(h + 1) * d].T / math.sqrt(d)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            outs.append(p @ v[:, h * d:(h + 1) * d])
        kc = k.reshape(-1, H, d)
        assert np.allclose(final["k_cache"][layer][0], kc, rtol=1e-12, atol=1e-12)
        x = np.concatenate(outs, axis=1)
    assert np.allclose(final["out"], x, rtol=1e-12, atol=1e-12)


def _first_masked(is_masked, prompt_len, L):
    gen = np.flatnonzero(is_masked[prompt_len:])
    return prompt_len + int(gen[0]) if gen.size else L


def _replay_masks(recs, w):
    """is_masked before every step, rebuilt from the records' unmask decisions."""
    im = np.zeros(w.seq_len, np.uint8)
    im[w.prompt_len:] = 1
    out = []
    for r in recs:
        out.append(im.copy())
        for u in r["unmask_rows"]:
            if u >= 0:
                im[r["row_pos"][u]] = 0
    return out


def test_sliding_window_invariants():
    # EntropyCache, section 5: the same skipping rule under a sliding window; the
    # window starts at the first still-masked position and holds W positions
    width = 12
    recs, final = otraj.run(W, 5, policy=("sliding", width))
    masks = _replay_masks(recs, W)
    for t, (r, im) in enumerate(zip(recs, masks)):
        lo = _first_masked(im, W.prompt_len, W.seq_len)
        assert r["window"] == (lo, min(lo + width, W.seq_len))
        want = np.flatnonzero(im[lo:lo + width]) + lo  # its masked positions, ascending
        assert np.array_equal(r["row_pos"], want)
        if t > 0 and not r["full"]:
            # the partial forward recomputes the masked positions of this window
            assert set(want.tolist()) <= set(r["idx"].tolist())
    assert final["is_masked"].sum() == 0


def test_multiblock_windows_are_whole_blocks():
    recs, _ = otraj.run(W, 6, policy=("multiblock", 2))
    masks = _replay_masks(recs, W)
    for r, im in zip(recs, masks):
        lo, hi = r["window"]
        first = _first_masked(im, W.prompt_len, W.seq_len)
        assert (lo - W.prompt_len) % W.block == 0 and lo <= first < lo + W.block
        assert hi == min(lo + 2 * W.block, W.seq_len)
        assert np.array_equal(r["row_pos"], np.flatnonzero(im[lo:hi]) + lo)


def test_window_rules_agree_when_the_window_covers_the_response():
    # a sliding window and a run of blocks as wide as the generated region see the
    # same masked positions at every step, so the trajectories are identical
    gen = W.seq_len - W.prompt_len
    a, fa = otraj.run(W, 7, policy=("sliding", gen))
    b, fb = otraj.run(W, 7, policy=("multiblock", gen // W.block))
    for ra, rb in zip(a, b):
        for key in ("full", "rows", "row_pos", "unmask_rows", "refresh", "idx_next"):
            assert np.array_equal(ra[key], rb[key]), key
    assert np.array_equal(fa["tokens"], fb["tokens"])
