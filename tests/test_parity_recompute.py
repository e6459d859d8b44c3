"""GPU recompute index set (ec_build_recompute_set) against the oracle, bit-exact,
on the workloads' decode states and on unstructured states with ragged
sequence lengths, every refresh pattern and k from 0 to beyond L."""
import numpy as np
import pytest

from entropy_gated_kv_decode_b300 import synth
from gpu_helpers import native, run_recompute_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "single_seq", "batched", "long_ctx", "trajectory"])
def test_workload_states(orc, name):
    nat = native()
    w = synth.WORKLOADS[name]
    st = synth.make_state(np.random.default_rng(0), w)
    refresh = np.zeros(w.batch, np.uint8)
    refresh[::3] = 1 if w.batch > 1 else 0
    g_idx, g_cnt = run_recompute_gpu(nat, st.is_masked, st.decode_step, refresh, st.block_lo,
                                     st.block_hi, w.k)
    o_idx, o_cnt = orc.recompute_set(st.is_masked, st.decode_step, refresh, st.block_lo,
                                     st.block_hi, w.k)
    assert np.array_equal(g_cnt, o_cnt)
    assert np.array_equal(g_idx, o_idx)
    for b in range(w.batch):
        if not refresh[b]:
            assert o_cnt[b] == w.r_max  # masked block + k most recent


@pytest.mark.parametrize("L", [1, 5, 1000, 1023, 1024, 1025, 3000, 8192, 10001])
@pytest.mark.parametrize("k", [0, 1, 16, 5000])
def test_random_states(orc, L, k):
    nat = native()
    rng = np.random.default_rng(L * 7 + k)
    B = 5
    im, ds = synth.random_state(rng, B, L, max_step=max(2, L // 8))
    refresh = np.array([0, 1, 0, 0, 1], np.uint8)
    lo = int(rng.integers(0, L))
    hi = int(rng.integers(lo, L + 1))
    g_idx, g_cnt = run_recompute_gpu(nat, im, ds, refresh, lo, hi, k)
    o_idx, o_cnt = orc.recompute_set(im, ds, refresh, lo, hi, k)
    assert np.array_equal(g_cnt, o_cnt)
    assert np.array_equal(g_idx, o_idx)


def test_many_ties_and_wide_step_range(orc):
    nat = native()
    rng = np.random.default_rng(99)
    B, L = 4, 4096
    im = np.zeros((B, L), np.uint8)
    ds = np.zeros((B, L), np.int32)
    ds[0] = 7                                        # every position decoded at the same step
    ds[1] = rng.integers(0, 2**31 - 1, size=L)       # huge step values
    ds[2, :] = -1                                    # nothing decoded
    ds[3] = rng.integers(0, 3, size=L)               # three big tie groups
    im[3, 100:200] = 1
    ds[3, 100:200] = -1
    for k in (1, 17, 1000, 4095, 4096):
        g = run_recompute_gpu(nat, im, ds, np.zeros(B, np.uint8), 50, 300, k)
        o = orc.recompute_set(im, ds, np.zeros(B, np.uint8), 50, 300, k)
        assert np.array_equal(g[1], o[1]) and np.array_equal(g[0], o[0]), k
