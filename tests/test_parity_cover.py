"""GPU attention with COVER's dual view (ec_selective_attention_cover) against the
oracle: the write-back of the non-seed rows bit-exact (seed positions keep the
previous K/V), outputs at the bf16 attention bounds (2e-2 relative / 1e-2
absolute elementwise, 2e-2 per-row relative Frobenius).  Every output row is
compared."""
import math

import numpy as np
import pytest
import torch

from entropy_gated_kv_decode_b300 import synth
from gpu_helpers import attention_close, dev, host, native

pytestmark = pytest.mark.gpu


def run_cover(orc, w, idx, cnt, seed, r_max, std=None, seed_rng=0):
    nat = native()
    a = synth.make_attention(np.random.default_rng(seed_rng), w, r_max, std)
    scale = 1.0 / math.sqrt(w.head_dim)
    q, kn, vn, kc, vc = (dev(x) for x in (a.q, a.k_new, a.v_new, a.k_cache, a.v_cache))
    out = torch.zeros_like(q)
    ws = nat.new_workspace(nat.ec_attention_workspace_size(w.batch, w.seq_len, r_max, w.n_heads,
                                                           w.n_kv_heads, w.head_dim))
    nat.ec_selective_attention_cover(q, kn, vn, dev(idx), dev(cnt), dev(seed), kc, vc, out, scale,
                                     ws)
    assert nat.ec_read_device_status(ws) == 0
    kc_ref, vc_ref, ref = orc.attention_cover(a.q, a.k_new, a.v_new, a.k_cache, a.v_cache, idx,
                                              cnt, seed, scale)
    assert np.array_equal(host(kc), kc_ref), "K write-back differs"
    assert np.array_equal(host(vc), vc_ref), "V write-back differs"
    got = synth.bf16_bits_to_f32(host(out)).astype(np.float64)
    for b in range(w.batch):
        assert not got[b, cnt[b]:].any()  # rows past count are left untouched
        attention_close(got[b, :cnt[b]], ref[b, :cnt[b]], True)
    return got


def _workload_set(orc, w):
    st = synth.make_state(np.random.default_rng(0), w)
    idx, cnt = orc.recompute_set(st.is_masked, st.decode_step, np.zeros(w.batch, np.uint8),
                                 st.block_lo, st.block_hi, w.k)
    return st, idx, cnt


@pytest.mark.parametrize("name,n_seeds", [("single_seq", 4), ("batched", 8), ("long_ctx", 16)])
@pytest.mark.parametrize("sharp", [False, True])
def test_workloads_with_seeds_among_the_recent_tokens(orc, name, n_seeds, sharp):
    w = synth.WORKLOADS[name]
    st, idx, cnt = _workload_set(orc, w)
    seed = synth.cover_seeds(np.random.default_rng(1), st.is_masked, idx, cnt, w.r_max, n_seeds)
    assert seed.sum() == w.batch * n_seeds
    run_cover(orc, w, idx, cnt, seed, w.r_max, std=1.0 if sharp else None)


@pytest.mark.parametrize("L,H,Hkv,d", [(1, 4, 4, 64), (129, 8, 2, 128), (300, 7, 1, 64),
                                       (2049, 14, 2, 128)])
def test_ragged_lengths_random_seeds(orc, L, H, Hkv, d):
    w = synth.scaled(synth.WORKLOADS["batched"], batch=3, seq_len=L, n_heads=H, n_kv_heads=Hkv,
                     head_dim=d, qkv_std=1.0)
    rng = np.random.default_rng(L + H)
    r_max = min(L, 150)
    cnt = np.array([r_max, max(0, r_max // 3), 1], np.int32)
    idx = synth.random_index_set(rng, w.batch, L, cnt, stride=r_max + 5)
    seed = (rng.random((w.batch, r_max)) < 0.3).astype(np.uint8)
    seed[2, 0] = 1  # a one-row sequence whose only row is a seed
    run_cover(orc, w, idx, cnt, seed, r_max, seed_rng=L)


def test_full_fresh_tiles_with_a_seed_inside(orc):
    # 256 consecutive recomputed positions (two whole fresh tiles): one tile holds a
    # seed, so it is patched row by row; the other comes in as one box
    w = synth.scaled(synth.WORKLOADS["single_seq"], seq_len=640, n_heads=8, n_kv_heads=8,
                     qkv_std=1.0)
    idx = np.arange(128, 384, dtype=np.int32)[None, :]
    cnt = np.array([256], np.int32)
    seed = np.zeros((1, 256), np.uint8)
    seed[0, [5, 77]] = 1
    run_cover(orc, w, idx, cnt, seed, 256)


def test_every_position_recomputed_with_seeds(orc):
    # count == L: the dense path is not taken, seeds keep their cached K/V
    w = synth.scaled(synth.WORKLOADS["single_seq"], seq_len=640, n_heads=8, n_kv_heads=8,
                     qkv_std=1.0)
    L = w.seq_len
    idx = np.arange(L, dtype=np.int32)[None, :]
    cnt = np.array([L], np.int32)
    seed = (np.random.default_rng(3).random((1, L)) < 0.05).astype(np.uint8)
    run_cover(orc, w, idx, cnt, seed, L)


def test_no_seed_equals_the_plain_call_bit_for_bit(orc):
    nat = native()
    w = synth.WORKLOADS["batched"]
    st, idx, cnt = _workload_set(orc, w)
    a = synth.make_attention(np.random.default_rng(4), w, w.r_max)
    scale = 1.0 / math.sqrt(w.head_dim)
    outs = []
    for cover in (False, True):
        q, kn, vn, kc, vc = (dev(x) for x in (a.q, a.k_new, a.v_new, a.k_cache, a.v_cache))
        out = torch.zeros_like(q)
        ws = nat.new_workspace(nat.ec_attention_workspace_size(w.batch, w.seq_len, w.r_max,
                                                               w.n_heads, w.n_kv_heads, w.head_dim))
        if cover:
            seed = torch.zeros((w.batch, w.r_max), dtype=torch.uint8, device="cuda")
            nat.ec_selective_attention_cover(q, kn, vn, dev(idx), dev(cnt), seed, kc, vc, out,
                                             scale, ws)
        else:
            nat.ec_selective_attention(q, kn, vn, dev(idx), dev(cnt), kc, vc, out, scale, ws)
        assert nat.ec_read_device_status(ws) == 0
        outs.append((host(out), host(kc), host(vc)))
    for x, y in zip(*outs):
        assert np.array_equal(x, y)
