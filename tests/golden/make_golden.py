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
    with open(os.path.join(HERE, "oracle_regression.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
