"""The oracle against its stored regression record (tests/golden/, written by
tests/golden/make_golden.py, which calls only oracle/).  The pages print no worked
numeric example of these quantities, so this record guards the oracle against silent
change; its independent pins are the closed forms of test_oracle_*.py."""
import json
import os

import numpy as np

from entropy_gated_kv_decode_b300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "oracle_regression.json")


def test_oracle_matches_its_regression_record(orc):
    with open(GOLDEN) as f:
        g = json.load(f)
    rs = g["row_stats"]
    h, c, t = orc.row_stats(np.array(rs["x"], np.float64))
    assert np.allclose(h, rs["entropy"], rtol=1e-12, atol=1e-14)
    assert np.allclose(c, rs["conf"], rtol=1e-12, atol=0)
    assert list(t) == rs["token"]

    d = g["decode_step"]
    w = synth.scaled(synth.WORKLOADS["tiny"], vocab=37, n_unmask=2, k=3, tau=1.0)
    st = synth.make_state(np.random.default_rng(7), w)
    logits = synth.make_logits(np.random.default_rng(8), w.n_rows, w.vocab, w.logits_dtype)
    hh, cc, tt = orc.row_stats(logits)
    res = orc.unmask_gate(cc, hh, tt, st.seq_row_offsets, st.row_pos, w.seq_len, w.n_unmask,
                          w.tau, st.step, st.is_masked, st.tokens, st.decode_step)
    assert np.asarray(res["unmask_rows"]).tolist() == d["unmask_rows"]
    assert np.allclose(res["max_entropy"], d["max_entropy"], rtol=1e-12, atol=1e-15)
    assert np.asarray(res["refresh"]).tolist() == d["refresh"]
    idx, cnt = orc.recompute_set(res["is_masked"], res["decode_step"], res["refresh"],
                                 st.block_lo, st.block_hi, w.k)
    assert cnt.tolist() == d["count"]
    assert idx[:, :int(cnt.max())].tolist() == d["idx"]


def test_variants_match_their_regression_record(orc):
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "make_golden", os.path.join(os.path.dirname(GOLDEN), "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    with open(GOLDEN) as f:
        g = json.load(f)["variants"]
    now = mg.variant_record()
    for key in ("simsd", "cover", "rms_norm", "rope", "cover_score"):
        assert np.allclose(np.array(now[key]), np.array(g[key]), rtol=1e-12, atol=1e-14,
                           equal_nan=True), key
    assert now["cover_seeds"] == g["cover_seeds"]
