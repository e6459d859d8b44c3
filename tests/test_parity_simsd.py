"""GPU KV write-back + attention under SimSD's temporal causal mask
(ec_selective_attention_simsd) against the oracle.  The write-back is bit-exact;
outputs meet the bf16 attention bounds of the unmasked kernel (2e-2 relative /
1e-2 absolute elementwise and a 2e-2 per-row relative Frobenius bound).  Every
output row is compared, except in the long-prompt case, which compares a seeded
sample of (sequence, row, head) outputs."""
import math

import numpy as np
import pytest
import torch

from entropy_gated_kv_decode_b300 import synth
from gpu_helpers import attention_close, dev, host, native

pytestmark = pytest.mark.gpu


def run_simsd(orc, w, section, tau, idx, cnt, r_max, seed=0, n_samples=0):
    nat = native()
    a = synth.make_attention(np.random.default_rng(seed), w, r_max)
    scale = 1.0 / math.sqrt(w.head_dim)
    q, kn, vn, kc, vc = (dev(x) for x in (a.q, a.k_new, a.v_new, a.k_cache, a.v_cache))
    out = torch.zeros_like(q)
    ws = nat.new_workspace(nat.ec_attention_workspace_size(w.batch, w.seq_len, r_max, w.n_heads,
                                                           w.n_kv_heads, w.head_dim))
    nat.ec_selective_attention_simsd(q, kn, vn, dev(idx), dev(cnt), dev(section), dev(tau), kc, vc,
                                     out, scale, ws)
    status = nat.ec_read_device_status(ws)
    kc_ref, vc_ref = orc.scatter_kv(a.k_new, a.v_new, idx, cnt, a.k_cache, a.v_cache)
    assert np.array_equal(host(kc), kc_ref), "K write-back differs"
    assert np.array_equal(host(vc), vc_ref), "V write-back differs"
    got = synth.bf16_bits_to_f32(host(out)).astype(np.float64)
    for b in range(w.batch):  # rows past count are left untouched
        assert not got[b, cnt[b]:].any()
    if n_samples:
        rng = np.random.default_rng(seed + 1)
        bs = rng.integers(0, w.batch, n_samples)
        rs = np.array([rng.integers(0, max(1, cnt[b])) for b in bs])
        keep = cnt[bs] > 0
        smp = np.stack([bs, rs, rng.integers(0, w.n_heads, n_samples)], axis=1)[keep]
        ref = orc.attention_simsd(a.q, kc_ref, vc_ref, idx, cnt, section, tau, scale, samples=smp)
        attention_close(got[smp[:, 0], smp[:, 1], smp[:, 2]], ref, True)
    else:
        ref = orc.attention_simsd(a.q, kc_ref, vc_ref, idx, cnt, section, tau, scale)
        for b in range(w.batch):
            attention_close(got[b, :cnt[b]], ref[b, :cnt[b]], True)
    return status, got


def test_simsd_verification_workload(orc):
    w = synth.SIMSD
    section, tau, idx, cnt = synth.make_simsd_layout(np.random.default_rng(0), w.batch,
                                                     w.prompt_len, w.block)
    status, _ = run_simsd(orc, w, section, tau, idx, cnt, 2 * w.block)
    assert status == 0


@pytest.mark.parametrize("prompt,blk,H,Hkv,d", [(276, 12, 7, 1, 64), (0, 100, 8, 2, 128),
                                                (1, 200, 4, 4, 128), (900, 64, 28, 4, 128)])
def test_ragged_layouts_with_prompt_queries(orc, prompt, blk, H, Hkv, d):
    # the query rows: every data and mask position plus some prompt positions, and
    # sequences with fewer rows (a shorter index set)
    L = prompt + 2 * blk
    w = synth.scaled(synth.SIMSD, batch=3, seq_len=L, prompt_len=prompt, block=blk, n_heads=H,
                     n_kv_heads=Hkv, head_dim=d)
    rng = np.random.default_rng(L + H)
    section, tau, _, _ = synth.make_simsd_layout(rng, w.batch, prompt, blk)
    n_prompt = min(prompt, 40)
    r_max = n_prompt + 2 * blk
    idx = np.full((w.batch, r_max + 3), -1, np.int32)
    cnt = np.zeros(w.batch, np.int32)
    for b in range(w.batch):
        rows = np.arange(prompt, L)
        if n_prompt:
            rows = np.concatenate([rng.choice(prompt, n_prompt, replace=False), rows])
        if b == 1:
            rows = rng.choice(rows, len(rows) // 3, replace=False)
        rows = np.sort(rows)
        idx[b, :len(rows)] = rows
        cnt[b] = len(rows)
    status, _ = run_simsd(orc, w, section, tau, idx, cnt, r_max, seed=L)
    assert status == 0


def test_long_prompt_split_over_ctas(orc):
    # one sequence whose keys are cut over many CTAs: prompt queries see nothing in
    # the pieces that cover only the response sections
    prompt, blk = 8192, 512
    L = prompt + 2 * blk
    w = synth.scaled(synth.SIMSD, batch=1, seq_len=L, prompt_len=prompt, block=blk, n_heads=16,
                     n_kv_heads=16, head_dim=128)
    rng = np.random.default_rng(5)
    section, tau, _, _ = synth.make_simsd_layout(rng, 1, prompt, blk)
    rows = np.sort(np.concatenate([rng.choice(prompt, 64, replace=False), np.arange(prompt, L)]))
    idx = rows[None].astype(np.int32)
    cnt = np.array([len(rows)], np.int32)
    status, _ = run_simsd(orc, w, section, tau, idx, cnt, len(rows), seed=6, n_samples=768)
    assert status == 0


def test_prompt_only_layout_equals_unmasked_attention(orc):
    # every key visible to every query: the masked kernel takes the unmasked
    # kernel's arithmetic, so the outputs agree bit for bit
    nat = native()
    w = synth.WORKLOADS["batched"]
    rng = np.random.default_rng(3)
    r_max = w.r_max
    cnt = np.full(w.batch, r_max, np.int32)
    idx = synth.random_index_set(rng, w.batch, w.seq_len, cnt, r_max)
    a = synth.make_attention(rng, w, r_max)
    scale = 1.0 / math.sqrt(w.head_dim)
    outs = []
    for masked in (False, True):
        q, kn, vn, kc, vc = (dev(x) for x in (a.q, a.k_new, a.v_new, a.k_cache, a.v_cache))
        out = torch.zeros_like(q)
        ws = nat.new_workspace(nat.ec_attention_workspace_size(w.batch, w.seq_len, r_max,
                                                               w.n_heads, w.n_kv_heads, w.head_dim))
        if masked:
            zeros8 = torch.zeros((w.batch, w.seq_len), dtype=torch.uint8, device="cuda")
            zeros32 = torch.zeros((w.batch, w.seq_len), dtype=torch.int32, device="cuda")
            nat.ec_selective_attention_simsd(q, kn, vn, dev(idx), dev(cnt), zeros8, zeros32, kc, vc,
                                             out, scale, ws)
        else:
            nat.ec_selective_attention(q, kn, vn, dev(idx), dev(cnt), kc, vc, out, scale, ws)
        assert nat.ec_read_device_status(ws) == 0
        outs.append(host(out))
    assert np.array_equal(outs[0], outs[1])


def test_bad_labels_raise_the_status_bit_and_hide_keys(orc):
    # a section value 3 on a key and a step label 0 on a query position: the key is
    # hidden, the query's row is zero, EC_DEV_BAD_LABEL is raised
    nat = native()
    w = synth.scaled(synth.SIMSD, batch=2, seq_len=300, prompt_len=260, block=20, n_heads=8,
                     n_kv_heads=2, head_dim=128)
    rng = np.random.default_rng(9)
    section, tau, idx, cnt = synth.make_simsd_layout(rng, w.batch, 260, 20)
    bad_key = 150
    section[0, bad_key] = 3
    bad_query = int(np.flatnonzero(idx[1] == 290)[0])
    tau[1, 290] = 0
    a = synth.make_attention(rng, w, 40)
    scale = 1.0 / math.sqrt(w.head_dim)
    q, kn, vn, kc, vc = (dev(x) for x in (a.q, a.k_new, a.v_new, a.k_cache, a.v_cache))
    out = torch.zeros_like(q)
    ws = nat.new_workspace(nat.ec_attention_workspace_size(w.batch, w.seq_len, 40, w.n_heads,
                                                           w.n_kv_heads, w.head_dim))
    nat.ec_selective_attention_simsd(q, kn, vn, dev(idx), dev(cnt), dev(section), dev(tau), kc, vc,
                                     out, scale, ws)
    assert nat.ec_read_device_status(ws) == nat.DEV_BAD_LABEL
    got = synth.bf16_bits_to_f32(host(out)).astype(np.float64)
    assert not got[1, bad_query].any()
    # sequence 0 matches the oracle with the bad key's section read as hidden: give
    # it a data label no query's window holds (above every step label)
    kc_ref, vc_ref = orc.scatter_kv(a.k_new, a.v_new, idx, cnt, a.k_cache, a.v_cache)
    sec_ref, tau_ref = section.copy(), tau.copy()
    sec_ref[0, bad_key], tau_ref[0, bad_key] = 1, 10**6
    ref = orc.attention_simsd(a.q, kc_ref, vc_ref, idx, cnt, sec_ref, np.maximum(tau_ref, 1), scale)
    attention_close(got[0], ref[0], True)


def test_rope_copy_gives_a_slot_its_data_tokens_rotation(orc):
    # item 3 (RoPE copy): the oracle side pairs each slot with the data token of the
    # same step label and takes that token's position; the product maps positions
    # by the layout (slot P + B + k -> P + k)
    from entropy_gated_kv_decode_b300 import simsd
    from oracle import layer as olayer
    nat = native()
    rng = np.random.default_rng(12)
    P, blk, H, Hkv, d = 1000, 8, 4, 2, 128
    section, tau, idx, cnt = synth.make_simsd_layout(rng, 3, P, blk)
    want = idx.copy()
    for b in range(3):
        for r in range(cnt[b]):
            p = idx[b, r]
            if section[b, p] == 2:
                data = [j for j in range(P, P + blk) if section[b, j] == 1 and tau[b, j] == tau[b, p]]
                want[b, r] = data[0]
    rope_pos = simsd.rope_positions(idx, cnt, P, blk)
    assert np.array_equal(rope_pos, want)
    q = synth.f32_to_bf16_bits(rng.standard_normal((3, 2 * blk, H, d), dtype=np.float32))
    k = synth.f32_to_bf16_bits(rng.standard_normal((3, 2 * blk, Hkv, d), dtype=np.float32))
    q[:, blk:] = q[:, :blk]  # each slot row the same vectors as its section-order data row
    k[:, blk:] = k[:, :blk]
    qd, kd = dev(q), dev(k)
    ws = nat.new_workspace(256)
    nat.ec_rope(qd, kd, dev(rope_pos), dev(cnt), P + 2 * blk, 500000.0, ws)
    got_q = synth.bf16_bits_to_f32(host(qd)).astype(np.float64)
    for b in range(3):
        ref = olayer.rope(q[b], want[b], 500000.0)
        assert np.all(np.abs(got_q[b] - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)
    # slot row k and data row k were equal and now sit at one rotary position
    assert np.array_equal(host(qd)[:, blk:], host(qd)[:, :blk])
    assert np.array_equal(host(kd)[:, blk:], host(kd)[:, :blk])
