"""GPU KV write-back + selective bidirectional attention (ec_selective_attention)
against the oracle.  The write-back must be bit-exact; outputs within 1e-4 for
float32 and 2e-2 relative / 1e-2 absolute for bf16 (plus a per-row relative
Frobenius bound, since the workloads' N(0, 1/sqrt(d)) operands give outputs of
magnitude ~1e-2).  Every output row is compared, at every workload's full size
(the oracle runs its rows on all host cores)."""
import math

import numpy as np
import pytest
import torch

from entropy_gated_kv_decode_b300 import synth
from gpu_helpers import attention_close, dev, host, native

pytestmark = pytest.mark.gpu


def run_case(orc, w, idx, cnt, r_max, std=None, seed=0):
    nat = native()
    rng = np.random.default_rng(seed)
    a = synth.make_attention(rng, w, r_max, std)
    scale = 1.0 / math.sqrt(w.head_dim)
    q, kn, vn, kc, vc = (dev(x) for x in (a.q, a.k_new, a.v_new, a.k_cache, a.v_cache))
    out = torch.zeros_like(q)
    ws = nat.new_workspace(nat.ec_attention_workspace_size(w.batch, w.seq_len, r_max, w.n_heads,
                                                           w.n_kv_heads,
                                                           w.head_dim))
    nat.ec_selective_attention(q, kn, vn, dev(idx), dev(cnt), kc, vc, out, scale, ws)
    assert nat.ec_read_device_status(ws) == 0
    kc_ref, vc_ref = orc.scatter_kv(a.k_new, a.v_new, idx, cnt, a.k_cache, a.v_cache)
    assert np.array_equal(host(kc), kc_ref), "K write-back differs"
    assert np.array_equal(host(vc), vc_ref), "V write-back differs"
    got = host(out)
    bf16 = w.attn_dtype == synth.BF16
    got64 = synth.bf16_bits_to_f32(got).astype(np.float64) if bf16 else got.astype(np.float64)
    for b in range(w.batch):  # rows past count are left untouched
        assert not got64[b, cnt[b]:].any()
    ref = orc.attention(a.q, kc_ref, vc_ref, cnt, scale)
    for b in range(w.batch):
        attention_close(got64[b, :cnt[b]], ref[b, :cnt[b]], bf16)


def _workload_index_set(orc, w):
    st = synth.make_state(np.random.default_rng(0), w)
    return orc.recompute_set(st.is_masked, st.decode_step, np.zeros(w.batch, np.uint8),
                             st.block_lo, st.block_hi, w.k)


@pytest.mark.parametrize("name", ["tiny", "single_seq", "batched", "long_ctx"])
@pytest.mark.parametrize("sharp", [False, True])
def test_workloads(orc, name, sharp):
    w = synth.WORKLOADS[name]
    idx, cnt = _workload_index_set(orc, w)
    assert (cnt == w.r_max).all()
    run_case(orc, w, idx, cnt, w.r_max, std=1.0 if sharp else None)


@pytest.mark.parametrize("L,H,Hkv,d", [(1, 4, 4, 64), (129, 8, 2, 128), (300, 7, 1, 64),
                                       (1000, 4, 4, 128), (2049, 14, 2, 128)])
@pytest.mark.parametrize("dt", [synth.BF16, synth.F32])
def test_ragged_lengths_and_head_groups(orc, L, H, Hkv, d, dt):
    w = synth.scaled(synth.WORKLOADS["batched"], batch=3, seq_len=L, n_heads=H, n_kv_heads=Hkv,
                     head_dim=d, attn_dtype=dt, qkv_std=1.0)
    rng = np.random.default_rng(L + H)
    r_max = min(L, 150)
    cnt = np.array([r_max, max(0, r_max // 3), 1 if L > 0 else 0], np.int32)
    idx = synth.random_index_set(rng, w.batch, L, cnt, stride=r_max + 5)
    run_case(orc, w, idx, cnt, r_max, seed=L)


def test_full_refresh_every_row_recomputed(orc):
    w = synth.scaled(synth.WORKLOADS["single_seq"], seq_len=640, n_heads=8, n_kv_heads=8,
                     qkv_std=1.0)
    L = w.seq_len
    idx = np.arange(L, dtype=np.int32)[None, :]
    cnt = np.array([L], np.int32)
    run_case(orc, w, idx, cnt, L)


def test_zero_rows(orc):
    w = synth.scaled(synth.WORKLOADS["single_seq"], seq_len=256, n_heads=4, n_kv_heads=4)
    idx = np.full((1, 8), -1, np.int32)
    run_case(orc, w, idx, np.zeros(1, np.int32), 8)


@pytest.mark.parametrize("batch,L,H,r", [(1, 2048, 4, 48), (1, 1024, 32, 48), (2, 512, 32, 100),
                                         (1, 1100, 4, 130)])
def test_few_units(orc, batch, L, H, r):
    # few units (4 to 64), each a whole unit on one CTA; the last case also has a
    # ragged key tile and a partial second row tile
    w = synth.scaled(synth.WORKLOADS["single_seq"], batch=batch, seq_len=L, n_heads=H,
                     n_kv_heads=H, qkv_std=1.0)
    rng = np.random.default_rng(L + H + r)
    cnt = np.full(batch, r, np.int32)
    idx = synth.random_index_set(rng, batch, L, cnt, stride=r)
    run_case(orc, w, idx, cnt, r, seed=L + r)
