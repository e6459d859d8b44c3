"""float64 oracle of a whole synthetic denoising trajectory with EntropyCache.

TEST INFRASTRUCTURE, like the rest of this package: only the tests, the smoke
check and the CPU-baseline leg of the benchmark use it.

EntropyCache, Italian summary, "Algoritmo di Funzionamento" steps 1-3 and the
Arabic technical summary, "Algorithm workflow" phases 1-3: at every step the
model runs a full forward (step 0, or when the previous step's gate fired) or a
partial one over the recompute set (the masked positions of the active block
and the k most recently decoded positions); the new tokens are decoded from
the step's logits, the max entropy E of the unmasked rows is compared with tau,
and the decode-time log is updated.

The steps are the oracle's own functions (row_stats, unmask_gate,
recompute_set; embed_rows, projection, scatter_kv, attention), composed in the
pages' order.  The workload's block schedule, starting state, weights and
logits come from the shared seeded generator.

Decoding policies (EntropyCache, Italian summary, section 5 "Generalità": the
entropy-based skipping applies to other decoding strategies, sliding windows and
blocks).  The positions a step may unmask, and the "currently masked" part of the
next recompute set, lie in the step's window [lo, hi):
  ("block",)          the workload's block schedule (blocks left to right);
  ("sliding", W)      lo = the first still-masked generated position, hi = lo + W;
  ("multiblock", nb)  lo = the start of the block holding the first still-masked
                      position, hi = lo + nb blocks;
hi clamped to L.  With the last two, a step's logits rows are the first c rows of
a W-row (nb-block) draw, c = the masked positions in its window.
"""
from __future__ import annotations

import math

import numpy as np

from entropy_gated_kv_decode_b300 import synth

from . import attention, embed_rows, projection, recompute_set, row_stats, scatter_kv, unmask_gate
from . import layer as olayer


def _widen(a):
    return synth.bf16_bits_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a


def window(w: synth.Workload, policy, t: int, is_masked: np.ndarray) -> tuple[int, int]:
    """The window [lo, hi) of step t under ``policy`` (see the module notes)."""
    if policy[0] == "block":
        return synth.trajectory_block(w, t)
    gen = np.flatnonzero(is_masked[0, w.prompt_len:])
    first = w.prompt_len + int(gen[0]) if gen.size else w.seq_len
    if policy[0] == "sliding":
        lo, width = first, policy[1]
    elif policy[0] == "multiblock":
        lo = w.prompt_len + (first - w.prompt_len) // w.block * w.block
        width = policy[1] * w.block
    else:
        raise ValueError(f"unknown policy {policy}")
    return lo, min(lo + width, w.seq_len)


def window_rows(w: synth.Workload, policy) -> int:
    """Rows of every step's logits draw under a window policy."""
    return policy[1] if policy[0] == "sliding" else policy[1] * w.block


def run(w: synth.Workload, seed: int, n_steps: int | None = None, logits_of_step=None,
        layers: int = 0, policy=("block",)):
    """Decisions (and, with ``layers`` > 0, the float64 forward of that many
    synthetic layers) of the first n_steps steps.  Returns a list of per-step
    dicts and the final state; with layers > 0 also the float64 K/V caches and
    the last forward's output rows."""
    n_steps = w.n_steps if n_steps is None else n_steps
    L, n, k, tau = w.seq_len, w.n_unmask, w.k, w.tau
    H, d = w.n_heads, w.head_dim
    hid = H * d
    if logits_of_step is None:
        if policy[0] == "block":
            rows_per_step = synth.trajectory_rows_per_step(w)

            def logits_of_step(t):
                return synth.trajectory_logits(seed, t, rows_per_step[t], w.vocab)
        else:
            def logits_of_step(t):
                return synth.trajectory_window_logits(seed, t, window_rows(w, policy), w.vocab)
    st = synth.trajectory_start(seed, w)
    im, tk, ds = st.is_masked.copy(), st.tokens.copy(), st.decode_step.copy()
    if layers:
        table = synth.trajectory_embedding(seed, w.vocab, hid)
        if w.ffn:
            weights = [synth.trajectory_layer_weights(seed, l, hid, w.ffn) for l in range(layers)]
        else:
            weights = [_widen(synth.trajectory_weights(seed, l, hid, hid)) for l in range(layers)]
        kc = [np.zeros((1, L, H, d)) for _ in range(layers)]
        vc = [np.zeros((1, L, H, d)) for _ in range(layers)]
    full_next, idx_next, cnt_next = True, None, None
    records, out = [], None
    for t in range(n_steps):
        # ---- forward of step t ----
        if full_next:
            idx = np.arange(L, dtype=np.int32)[None, :]
            cnt = np.array([L], np.int32)
        else:
            idx, cnt = idx_next, cnt_next
        if layers:
            r = int(cnt[0])
            x = _widen(embed_rows(table, idx, cnt, tk, im, w.vocab, r)).reshape(r, hid)
            for l in range(layers):
                if w.ffn:  # a pre-norm block (oracle/layer.py)
                    lw = weights[l]
                    a = olayer.rms_norm(x, lw["g1"], w.norm_eps)
                    y = olayer.linear(a, lw["w_qkv"])
                    pos = idx[0, :r]
                    q = olayer.rope(y[:, :hid].reshape(r, H, d), pos, w.rope_theta).reshape(1, r, H, d)
                    kn = olayer.rope(y[:, hid:2 * hid].reshape(r, H, d), pos,
                                     w.rope_theta).reshape(1, r, H, d)
                    vn = y[:, 2 * hid:].reshape(1, r, H, d)
                    kc[l], vc[l] = scatter_kv(kn, vn, idx, cnt, kc[l], vc[l])
                    o = attention(q, kc[l], vc[l], cnt, 1.0 / math.sqrt(d)).reshape(r, hid)
                    x = olayer.linear(o, lw["w_o"], 1, x)
                    b = olayer.rms_norm(x, lw["g2"], w.norm_eps)
                    x = olayer.linear(olayer.linear(b, lw["w_gu"], 2), lw["w_down"], 1, x)
                    continue
                y = projection(x, weights[l])
                q = y[:, :hid].reshape(1, r, H, d)
                kn = y[:, hid:2 * hid].reshape(1, r, H, d)
                vn = y[:, 2 * hid:].reshape(1, r, H, d)
                kc[l], vc[l] = scatter_kv(kn, vn, idx, cnt, kc[l], vc[l])
                x = attention(q, kc[l], vc[l], cnt, 1.0 / math.sqrt(d)).reshape(r, hid)
            out = x
        # ---- decode and gate with step t's logits ----
        lo, hi = window(w, policy, t, im)
        pos_idx, pos_cnt = recompute_set(im, ds, np.zeros(1, np.uint8), lo, hi, 0)
        row_pos = pos_idx[0, :pos_cnt[0]]
        logits = logits_of_step(t)
        if policy[0] != "block":
            logits = logits[:row_pos.shape[0]]
        if logits.shape[0] != row_pos.shape[0]:
            raise ValueError("step logits do not match the masked rows of the block")
        h, c, tok = row_stats(logits)
        g = unmask_gate(c, h, tok, [0, len(row_pos)], row_pos, L, n, tau, t, im, tk, ds)
        im, tk, ds = g["is_masked"], g["tokens"], g["decode_step"]
        nlo, nhi = window(w, policy, t + 1, im)
        idx_next, cnt_next = recompute_set(im, ds, g["refresh"], nlo, nhi, k)
        records.append(dict(step=t, full=full_next, rows=int(cnt[0]), window=(lo, hi),
                            idx=idx[0, :cnt[0]].copy(),
                            row_pos=row_pos.copy(), unmask_rows=g["unmask_rows"][0].copy(),
                            token=tok, entropy=h, conf=c, max_entropy=float(g["max_entropy"][0]),
                            refresh=int(g["refresh"][0]),
                            idx_next=idx_next[0, :cnt_next[0]].copy()))
        full_next = bool(g["refresh"][0])
    final = dict(is_masked=im, tokens=tk, decode_step=ds)
    if layers:
        final.update(k_cache=kc, v_cache=vc, out=out)
    return records, final
