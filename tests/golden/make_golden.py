"""Writes oracle_regression.json: the float64 oracle's outputs on small seeded
inputs, a regression record of the oracle.  It calls only oracle/ (and the seeded
generators in synth.py, which hold none of the method's arithmetic).

The pages ("EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion
Language Models", its Italian, Arabic and Hindi summaries) print no worked numeric
example of the row statistics, the unmasking, the gate or the recompute set; the
numbers they print are end-to-end results on trained models.  The oracle's
independent pins are therefore the closed forms, hand-worked rows and invariants
of tests/test_oracle_*.py; this fixture only guards the oracle against silent
change.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from entropy_gated_kv_decode_b300 import synth  # noqa: E402


def variant_inputs():
    """Seeded inputs of the attention variants and the layer pieces (shared with
    tests/test_golden.py)."""
    rng = np.random.default_rng(2025)
    sec, tau, idx, cnt = synth.make_simsd_layout(rng, 1, 3, 2)  # L = 7
    q = rng.standard_normal((1, 4, 2, 4))
    kc = rng.standard_normal((1, 7, 1, 4))
    vc = rng.standard_normal((1, 7, 1, 4))
    kn = rng.standard_normal((1, 4, 1, 4))
    vn = rng.standard_normal((1, 4, 1, 4))
    seed = np.array([[0, 1, 0, 1]], np.uint8)
    x = rng.standard_normal((3, 8))
    g = rng.standard_normal(8)
    role = np.array([[1, 2, 3, 2]], np.uint8)       # COVER seed score: masked / candidate rows
    drafted = np.array([[0, 0, 0, 1, 0, 1, 0]], np.uint8)
    u = np.array([[0.5, 1.25, 2.0, 0.75]])
    return dict(sec=sec, tau=tau, idx=idx, cnt=cnt, q=q, kc=kc, vc=vc, kn=kn, vn=vn, seed=seed,
                x=x, g=g, role=role, drafted=drafted, u=u)


def variant_record():
    from oracle import layer
    v = variant_inputs()
    simsd = oracle.attention_simsd(v["q"], v["kc"], v["vc"], v["idx"], v["cnt"], v["sec"],
                                   v["tau"], 0.5)
    _, _, cover = oracle.attention_cover(v["q"], v["kn"], v["vn"], v["kc"], v["vc"], v["idx"],
                                         v["cnt"], v["seed"], 0.5)
    d_in, d_out, score, seeds = oracle.cover_seed_score(v["q"], v["kc"], v["idx"], v["cnt"],
                                                        v["role"], v["drafted"], v["u"], 0.5, 3)
    return {"simsd": simsd.tolist(), "cover": cover.tolist(),
            "cover_score": [d_in.tolist(), d_out.tolist(), score.tolist()],
            "cover_seeds": seeds.tolist(),
            "rms_norm": layer.rms_norm(v["x"], v["g"], 1e-5).tolist(),
            "rope": layer.rope(v["x"].reshape(3, 1, 8), [0, 5, 900], 10000.0).tolist()}


def main():
    rng = np.random.default_rng(2024)
    x = rng.standard_normal((6, 37)) * np.array([[0.3], [1.0], [3.0], [0.1], [8.0], [1.5]])
    x[2, 5] += 6.0
    x[4, [3, 20]] = x[4].max() + 1.0  # a tie: the lower index wins
    h, c, t = oracle.row_stats(x)
    w = synth.scaled(synth.WORKLOADS["tiny"], vocab=37, n_unmask=2, k=3, tau=1.0)
    st = synth.make_state(np.random.default_rng(7), w)
    logits = synth.make_logits(np.random.default_rng(8), w.n_rows, w.vocab, w.logits_dtype)
    hh, cc, tt = oracle.row_stats(logits)
    g = oracle.unmask_gate(cc, hh, tt, st.seq_row_offsets, st.row_pos, w.seq_len, w.n_unmask,
                           w.tau, st.step, st.is_masked, st.tokens, st.decode_step)
    idx, cnt = oracle.recompute_set(g["is_masked"], g["decode_step"], g["refresh"], st.block_lo,
                                    st.block_hi, w.k)
    out = {
        "row_stats": {"x": x.tolist(), "entropy": h.tolist(), "conf": c.tolist(),
                      "token": t.tolist()},
        "decode_step": {"workload": "tiny, vocab 37, n_unmask 2, k 3, tau 1.0, state seed 7, "
                                    "logits seed 8",
                        "unmask_rows": np.asarray(g["unmask_rows"]).tolist(),
                        "max_entropy": np.asarray(g["max_entropy"]).tolist(),
                        "refresh": np.asarray(g["refresh"]).tolist(),
                        "idx": idx[:, :int(cnt.max())].tolist(), "count": cnt.tolist()},
    }
    out["variants"] = variant_record()
    with open(os.path.join(HERE, "oracle_regression.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
