"""Prepared (validate-once) calls of the binding give the same results as the
direct calls, for all three entry points."""
import math

import numpy as np
import pytest
import torch

from entropy_gated_kv_decode_b300 import synth
from gpu_helpers import dev, host, native

pytestmark = pytest.mark.gpu


def test_prepared_calls_match_direct_calls():
    nat = native()
    w = synth.scaled(synth.WORKLOADS["batched"], batch=2, vocab=8192, seq_len=512,
                     prompt_len=128, block=64, active_block=2)
    rng = np.random.default_rng(5)
    st = synth.make_state(rng, w)
    logits = dev(synth.make_logits(rng, w.n_rows, w.vocab, w.logits_dtype))
    att = synth.make_attention(rng, w, w.r_max)
    B, L, N, n = w.batch, w.seq_len, w.n_rows, w.n_unmask

    def run(prepared):
        outs = [torch.empty(N, dtype=torch.int32, device="cuda"),
                torch.empty(N, device="cuda"), torch.empty(N, device="cuda"),
                torch.empty(B * n, dtype=torch.int32, device="cuda"),
                torch.empty(B, device="cuda"), torch.empty(B, dtype=torch.uint8, device="cuda")]
        state = [dev(st.is_masked.copy()), dev(st.tokens.copy()), dev(st.decode_step.copy())]
        ws = nat.new_workspace(nat.ec_decode_workspace_size(N, B))
        args = (logits, dev(st.seq_row_offsets), dev(st.row_pos), L, n, w.tau, st.step,
                *outs, *state, ws)
        idx = torch.empty((B, L), dtype=torch.int32, device="cuda")
        cnt = torch.empty(B, dtype=torch.int32, device="cuda")
        rargs = (state[0], state[2], outs[5], st.block_lo, st.block_hi, w.k, idx, cnt)
        q, kn, vn, kc, vc = (dev(x) for x in (att.q, att.k_new, att.v_new, att.k_cache,
                                              att.v_cache))
        out = torch.zeros_like(q)
        wsa = nat.new_workspace(nat.ec_attention_workspace_size(B, L, w.r_max, w.n_heads, w.n_kv_heads,
                                                                w.head_dim))
        aargs = (q, kn, vn, idx, cnt, kc, vc, out, 1 / math.sqrt(w.head_dim), wsa)
        if prepared:
            d = nat.prepare_decode_step(*args)
            d.set_step(st.step)
            d()
            nat.prepare_build_recompute_set(*rargs)()
            nat.prepare_selective_attention(*aargs)()
        else:
            nat.ec_decode_step(*args)
            nat.ec_build_recompute_set(*rargs)
            nat.ec_selective_attention(*aargs)
        torch.cuda.synchronize()
        return [host(t) for t in outs + state + [idx, cnt, out, kc]]

    for a, b in zip(run(False), run(True)):
        assert np.array_equal(a, b)
