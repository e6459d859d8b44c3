"""GPU pre-norm layer pieces (ec_rms_norm, ec_rope, ec_linear) against the float64
oracle (oracle/layer.py), and a small trajectory of pre-norm layers against the
oracle's forward.

Bounds, from the arithmetic: every output is rounded once to bf16 (relative
2^-9; 2^-8 is used), float32 sums add hidden * 2^-24 * sum|terms|, the rotary
angles are exact in double and rounded to float32 (2^-24), silu uses __expf
(a few ulp)."""
import numpy as np
import pytest
import torch

import oracle.trajectory as otraj
from entropy_gated_kv_decode_b300 import synth
from gpu_helpers import dev, host, native
from oracle import layer as olayer

pytestmark = pytest.mark.gpu

U = 2.0 ** -8


def bf(rng, shape, scale=1.0):
    return synth.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(scale))


def wide(t):
    return synth.bf16_bits_to_f32(host(t)).astype(np.float64)


@pytest.mark.parametrize("B,R,hidden,cnt", [(2, 5, 4096, [5, 2]), (1, 3, 8, [3]), (3, 130, 128, [130, 0, 77])])
def test_rms_norm(B, R, hidden, cnt):
    nat = native()
    rng = np.random.default_rng(hidden + R)
    x = bf(rng, (B, R, hidden), 3.0)
    g = synth.f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(hidden)).astype(np.float32))
    y = torch.full((B, R, hidden), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = nat.new_workspace(256)
    count = np.array(cnt, np.int32)
    nat.ec_rms_norm(dev(x), dev(count), dev(g), 1e-5, y, ws)
    got = wide(y)
    ref = olayer.rms_norm(x, g, 1e-5)
    for b in range(B):
        c = cnt[b]
        assert np.all(np.abs(got[b, :c] - ref[b, :c]) <= U * np.abs(ref[b, :c]) + 1e-6)
        assert np.all(got[b, c:] == 7.0)


@pytest.mark.parametrize("H,Hkv,d,theta", [(32, 32, 128, 500000.0), (28, 4, 128, 10000.0), (4, 2, 64, 10000.0)])
def test_rope(H, Hkv, d, theta):
    nat = native()
    rng = np.random.default_rng(H + d)
    B, R, L = 2, 40, 8192
    q = bf(rng, (B, R, H, d))
    k = bf(rng, (B, R, Hkv, d))
    cnt = np.array([R, 17], np.int32)
    idx = synth.random_index_set(rng, B, L, cnt, R)
    idx[0, -1] = L - 1  # the largest angle
    qd, kd = dev(q), dev(k)
    ws = nat.new_workspace(256)
    nat.ec_rope(qd, kd, dev(idx), dev(cnt), L, theta, ws)
    assert nat.ec_read_device_status(ws) == 0
    for t, src in ((qd, q), (kd, k)):
        got = wide(t)
        for b in range(B):
            c = cnt[b]
            ref = olayer.rope(src[b, :c], idx[b, :c], theta)
            x = olayer.widen(src[b, :c])
            pair = np.sqrt(x[..., :d // 2] ** 2 + x[..., d // 2:] ** 2)
            tol = U * np.abs(ref) + 4e-7 * np.concatenate([pair, pair], axis=-1)
            assert np.all(np.abs(got[b, :c] - ref) <= tol)
            assert np.array_equal(host(t)[b, c:], src[b, c:])  # rows past count untouched


def _linear_bound(x, w, ref, mode):
    """Elementwise bound: bf16 rounding of the result plus float32 summation."""
    ax, aw = np.abs(olayer.widen(x)), np.abs(olayer.widen(w))
    n = ax.shape[-1]
    if mode == 2:
        f = w.shape[0] // 2
        g = olayer.widen(x) @ olayer.widen(w[:f]).T
        u = olayer.widen(x) @ olayer.widen(w[f:]).T
        sg, su = ax @ aw[:f].T, ax @ aw[f:].T
        acc = n * 2.0 ** -24 * (sg * np.abs(u) * 1.2 + np.abs(olayer.silu(g)) * su) + 1e-6 * np.abs(ref)
    else:
        acc = n * 2.0 ** -24 * (ax @ aw.T)
    return U * np.abs(ref) + 2 * acc + 1e-30


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("B,R,n_in,n_out,cnt", [(2, 100, 128, 256, [100, 31]), (1, 300, 512, 192, [300])])
def test_linear_small(mode, B, R, n_in, n_out, cnt):
    nat = native()
    rng = np.random.default_rng(mode * 10 + n_in)
    x = bf(rng, (B, R, n_in))
    w = bf(rng, (2 * n_out if mode == 2 else n_out, n_in), 1 / np.sqrt(n_in))
    res = bf(rng, (B, R, n_out))
    y = dev(res) if mode == 1 else torch.full((B, R, n_out), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = nat.new_workspace(256)
    count = np.array(cnt, np.int32)
    nat.ec_linear(dev(x), dev(count), dev(w), mode, y if mode == 1 else None, y, ws)
    got = wide(y)
    for b in range(B):
        c = cnt[b]
        ref = olayer.linear(x[b, :c], w, mode, res[b, :c])
        assert np.all(np.abs(got[b, :c] - ref) <= _linear_bound(x[b, :c], w, ref, mode))
        if mode == 1:
            assert np.array_equal(host(y)[b, c:], res[b, c:])
        else:
            assert np.all(got[b, c:] == 7.0)


@pytest.mark.parametrize("mode,n_in,n_out", [(2, 4096, 12288), (1, 12288, 4096), (1, 4096, 4096)])
def test_linear_full_size_sampled_rows(mode, n_in, n_out):
    # the trajectory model's MLP and output projection on 1024 rows; 12 rows checked
    nat = native()
    rng = np.random.default_rng(n_in + n_out + mode)
    R = 1024
    x = bf(rng, (1, R, n_in))
    w = bf(rng, (2 * n_out if mode == 2 else n_out, n_in), 1 / np.sqrt(n_in))
    res = bf(rng, (1, R, n_out))
    y = dev(res) if mode == 1 else torch.empty((1, R, n_out), dtype=torch.bfloat16, device="cuda")
    ws = nat.new_workspace(256)
    nat.ec_linear(dev(x), None, dev(w), mode, y if mode == 1 else None, y, ws)
    got = wide(y)
    rows = np.sort(rng.choice(R, 12, replace=False))
    ref = olayer.linear(x[0, rows], w, mode, res[0, rows])
    assert np.all(np.abs(got[0, rows] - ref) <= _linear_bound(x[0, rows], w, ref, mode))


SMALL = synth.scaled(synth.WORKLOADS["trajectory"], vocab=3000, seq_len=256, prompt_len=192,
                     block=16, n_heads=2, n_kv_heads=2, head_dim=64, n_layers=2, n_steps=32,
                     ffn=256, tau=2.5)


def test_prenorm_trajectory_small_model():
    from entropy_gated_kv_decode_b300.trajectory import Trajectory
    native()
    w = SMALL
    tr = Trajectory(w, seed=5, trace=True)
    tr.warm_up()
    recs = tr.run()
    torch.cuda.synchronize()
    ref, final = otraj.run(w, 5, layers=w.n_layers)
    assert [r.full for r in recs] == [o["full"] for o in ref]
    assert any(not r.full for r in recs)
    # caches: two layers of bf16 roundings at every op; a per-row relative
    # Frobenius bound of 4e-2 (about 8 roundings of 2^-9 per layer, added up)
    for layer in range(w.n_layers):
        for name, g in (("k", tr.k_cache[layer]), ("v", tr.v_cache[layer])):
            got = synth.bf16_bits_to_f32(host(g)).astype(np.float64)[0].reshape(w.seq_len, -1)
            want = (final["k_cache"] if name == "k" else final["v_cache"])[layer][0].reshape(w.seq_len, -1)
            num = np.linalg.norm(got - want, axis=1)
            den = np.linalg.norm(want, axis=1) + 1e-12
            assert np.max(num / den) <= 4e-2, f"layer {layer} {name} cache: {np.max(num / den)}"
    r = recs[-1].rows
    got = synth.bf16_bits_to_f32(host(tr.xa[0, :r])).astype(np.float64)
    want = final["out"]
    rel = np.linalg.norm(got - want, axis=1) / (np.linalg.norm(want, axis=1) + 1e-12)
    assert np.max(rel) <= 4e-2, f"output rows: {np.max(rel)}"
