"""Seeded cases for COVER's seed score, and the comparison of a float32 result
(GPU, or the kernels' items run on the host) with the float64 oracle.

Bounds, from the arithmetic: a score s = scale q.k is a float32 dot product of
exact bf16 products (error about D 2^-24 sum|q_e k_e| scale), each probability
takes one expf (a few ulp) and a normaliser summed in float32 over at most
(64 + key ranges) terms in sequence, so every probability, and every sum of
probabilities, is within about 1e-5 relative; 2e-4 relative plus 1e-6 absolute
is used for d_in, d_out and the score.  The seed ranking compares the float32
scores: it must be exactly the ranking of the result's own scores, and agree with
the oracle's ranking up to near ties (scores within 1e-3 relative)."""
import numpy as np

from entropy_gated_kv_decode_b300 import synth

RTOL, ATOL = 2e-4, 1e-6
TIE_RTOL = 1e-3
CANARY = 7.0


def own_ranking(score, idx, cand_rows, n_seed):
    """Seed positions by (score desc, position asc), NaN last, padded with -1."""
    keys = [(-(score[r] if score[r] == score[r] else -np.inf), int(idx[r]), int(idx[r]))
            for r in cand_rows]
    ranked = [k[2] for k in sorted(keys)][:n_seed]
    return ranked + [-1] * (n_seed - len(ranked))


def check(got, ref, idx, count, role, n_seed):
    d_in, d_out, score, seeds = got
    r_in, r_out, r_score, r_seeds = ref
    batch, r_max = role.shape
    for b in range(batch):
        c = int(min(max(count[b], 0), r_max))
        cand = np.array([r for r in range(c) if role[b, r] & 2], np.int64)
        other = np.setdiff1d(np.arange(r_max), cand)
        for name, x, y in (("d_in", d_in, r_in), ("d_out", d_out, r_out), ("score", score, r_score)):
            g, w = x[b, cand].astype(np.float64), y[b, cand]
            bad = np.abs(g - w) > RTOL * np.abs(w) + ATOL
            assert not bad.any(), f"{name} sequence {b} rows {cand[bad][:5]}: {g[bad][:5]} vs {w[bad][:5]}"
            assert np.all(x[b, other] == CANARY), f"{name} written outside the candidates"
        if n_seed == 0:
            continue
        assert seeds[b].tolist() == own_ranking(score[b], idx[b], cand, n_seed), \
            f"sequence {b}: seeds are not the ranking of the scores"
        n = min(n_seed, len(cand))
        assert np.all(seeds[b, n:] == -1) and np.all(r_seeds[b, n:] == -1)
        pos_row = {int(idx[b, r]): r for r in cand}
        want = np.sort(r_score[b, cand])[::-1][:n]
        have = np.array([r_score[b, pos_row[int(p)]] for p in seeds[b, :n]])
        assert np.all(np.abs(have - want) <= TIE_RTOL * np.abs(want) + ATOL), \
            f"sequence {b}: seed order departs from the oracle's beyond near ties"


def workload_case(orc, name, n_drafted, std=None, seed=0):
    w = synth.WORKLOADS[name]
    st = synth.make_state(np.random.default_rng(seed), w)
    idx, cnt = orc.recompute_set(st.is_masked, st.decode_step, np.zeros(w.batch, np.uint8),
                                 st.block_lo, st.block_hi, w.k)
    a = synth.make_attention(np.random.default_rng(seed + 1), w, w.r_max, std)
    role, drafted, u = synth.cover_score_inputs(np.random.default_rng(seed + 2), st.is_masked, idx,
                                                cnt, w.r_max, n_drafted)
    return a.q, a.k_cache, idx, cnt, role, drafted, u, 1.0 / np.sqrt(w.head_dim)


def ragged_case(rng, B, L, R, H, Hkv, D, std=1.0):
    q = synth.f32_to_bf16_bits(rng.standard_normal((B, R, H, D), dtype=np.float32) * np.float32(std))
    kc = synth.f32_to_bf16_bits(rng.standard_normal((B, L, Hkv, D), dtype=np.float32) * np.float32(std))
    cnt = np.array([min(R, L)] + [int(rng.integers(0, min(R, L) + 1)) for _ in range(B - 1)], np.int32)
    idx = synth.random_index_set(rng, B, L, cnt, stride=R + 3)
    role = rng.integers(0, 4, (B, R)).astype(np.uint8)
    drafted = (rng.random((B, L)) < 0.1).astype(np.uint8)
    u = rng.uniform(0, 5, (B, R)).astype(np.float32)
    return q, kc, idx, cnt, role, drafted, u, 1.0 / np.sqrt(D)
