"""GPU first-layer gather (ec_embed_rows, bit-exact) and Q/K/V projection
(ec_qkv_projection) against the float64 oracle.

Tolerance of the projection, derived from its arithmetic: the tensor cores
accumulate the hidden-length dot product in float32 (error at most about
hidden * 2^-24 * sum_e |x_e w_e|) and the result is rounded once to bf16
(relative error at most 2^-9); the test allows four times the first term plus
2^-8 |y|."""
import numpy as np
import pytest
import torch

from entropy_gated_kv_decode_b300 import synth
from gpu_helpers import dev, host, native

pytestmark = pytest.mark.gpu


def _bf16(rng, shape, std):
    return synth.f32_to_bf16_bits((rng.standard_normal(shape, dtype=np.float32) * np.float32(std)))


def _abs_bits(a):
    return (a & np.uint16(0x7FFF)).astype(np.uint16)


def run_projection(orc, batch, r_max, hidden, width, counts, seed=0, sample_rows=None):
    nat = native()
    rng = np.random.default_rng(seed)
    x = _bf16(rng, (batch, r_max, hidden), 1.0)
    w = _bf16(rng, (3 * width, hidden), 1.0 / np.sqrt(hidden))
    cnt = np.asarray(counts, np.int32)
    outs = [torch.full((batch, r_max, width), float("nan"), dtype=torch.bfloat16, device="cuda")
            for _ in range(3)]
    ws = nat.new_workspace(256)
    nat.ec_qkv_projection(dev(x), dev(cnt), dev(w), *outs, ws)
    assert nat.ec_read_device_status(ws) == 0
    got = np.concatenate([synth.bf16_bits_to_f32(host(o)).astype(np.float64) for o in outs], axis=-1)
    flat_x = x.reshape(batch * r_max, hidden)
    rows = [b * r_max + r for b in range(batch) for r in range(cnt[b])]
    if sample_rows is not None and len(rows) > sample_rows:
        rows = sorted(rng.choice(rows, size=sample_rows, replace=False).tolist())
    if rows:
        ref = orc.projection(flat_x, w, rows=rows)
        mag = orc.projection(_abs_bits(flat_x), _abs_bits(w), rows=rows)
        g = got.reshape(batch * r_max, 3 * width)[rows]
        tol = 4 * hidden * 2.0**-24 * mag + 2.0**-8 * np.abs(ref) + 1e-30
        assert np.all(np.abs(g - ref) <= tol), f"max excess {np.max(np.abs(g - ref) - tol)}"
    for b in range(batch):  # rows past count are left untouched
        assert np.isnan(got[b, cnt[b]:]).all()


def test_trajectory_full_refresh_shape(orc):
    # every position of a 1024-token sequence through a 4096 -> 3 x 4096 projection
    run_projection(orc, 1, 1024, 4096, 4096, [1024])


def test_trajectory_selective_shape(orc):
    # 46 recomputed rows in a buffer sized for 48
    run_projection(orc, 1, 48, 4096, 4096, [46])


@pytest.mark.parametrize("batch,r_max,hidden,width,counts", [
    (3, 130, 64, 64, [130, 0, 77]),
    (1, 1, 128, 64, [1]),
    (2, 300, 256, 384, [300, 129]),
    (1, 257, 192, 192, [256]),
    (2, 64, 512, 512, [64, 63]),
])
def test_ragged_shapes(orc, batch, r_max, hidden, width, counts):
    run_projection(orc, batch, r_max, hidden, width, counts, seed=r_max + width)


def test_no_count_means_every_row(orc):
    nat = native()
    rng = np.random.default_rng(3)
    x = _bf16(rng, (1, 70, 128), 1.0)
    w = _bf16(rng, (3 * 128, 128), 0.1)
    outs = [torch.zeros((1, 70, 128), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    ws = nat.new_workspace(256)
    nat.ec_qkv_projection(dev(x), None, dev(w), *outs, ws)
    got = np.concatenate([synth.bf16_bits_to_f32(host(o)).astype(np.float64) for o in outs], -1)
    ref = orc.projection(x.reshape(70, 128), w)
    assert np.allclose(got.reshape(70, 384), ref, rtol=2.0**-7, atol=1e-3)


@pytest.mark.parametrize("L,hidden,r_max", [(64, 64, 40), (1024, 4096, 1024), (300, 136, 250)])
def test_embed_rows_bit_exact(orc, L, hidden, r_max):
    nat = native()
    rng = np.random.default_rng(L)
    V, B = 1000, 2
    table = _bf16(rng, (V + 1, hidden), 1.0)
    tokens = rng.integers(0, V, size=(B, L)).astype(np.int32)
    is_masked = (rng.uniform(size=(B, L)) < 0.3).astype(np.uint8)
    cnt = np.array([r_max, r_max // 2], np.int32)
    idx = synth.random_index_set(rng, B, L, cnt, stride=L)
    x = torch.zeros((B, r_max, hidden), dtype=torch.bfloat16, device="cuda")
    ws = nat.new_workspace(256)
    nat.ec_embed_rows(dev(table), dev(idx), dev(cnt), dev(tokens), dev(is_masked), V, x, ws)
    assert nat.ec_read_device_status(ws) == 0
    ref = orc.embed_rows(table, idx, cnt, tokens, is_masked, V, r_max)
    assert np.array_equal(host(x), ref)
