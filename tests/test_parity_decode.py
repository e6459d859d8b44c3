"""GPU decode-and-gate step (ec_decode_step) against the float64 oracle, on the
seeded workloads at full size and on edge cases: ragged vocabularies, padded
row strides, -inf logits, exact ties, empty and short sequences."""
import numpy as np
import pytest

from entropy_gated_kv_decode_b300 import synth
from gpu_helpers import check_decode, native, run_decode_gpu, run_decode_oracle

pytestmark = pytest.mark.gpu

REPORT = []


def _case(orc, w, seed=0, **kw):
    nat = native()
    rng = np.random.default_rng(seed)
    st = synth.make_state(rng, w)
    logits = synth.make_logits(rng, w.n_rows, w.vocab, w.logits_dtype, w.near_uniform_frac)
    gpu = run_decode_gpu(nat, logits, st, w.n_unmask, w.tau, st.step, **kw)
    ref = run_decode_oracle(orc, logits, st, w.n_unmask, w.tau, st.step)
    excluded = check_decode(gpu, ref, st, w.n_unmask, w.tau, st.step)
    REPORT.append((w.name, seed, sorted(excluded)))
    assert len(excluded) <= max(1, w.batch // 4), f"too many excluded decisions: {excluded}"
    return gpu, ref, st


@pytest.mark.parametrize("name", ["tiny", "single_seq", "batched", "long_ctx"])
def test_workloads_full_size(orc, name):
    _case(orc, synth.WORKLOADS[name])


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_single_seq_other_seeds(orc, seed):
    _case(orc, synth.WORKLOADS["single_seq"], seed=seed)


@pytest.mark.parametrize("vocab", [1, 7, 9, 1000, 4099, 126463])
@pytest.mark.parametrize("dt", [synth.BF16, synth.F32])
def test_ragged_vocab(orc, vocab, dt):
    w = synth.scaled(synth.WORKLOADS["single_seq"], vocab=vocab, logits_dtype=dt, batch=3,
                     seq_len=256, prompt_len=64, block=16, active_block=4, n_unmask=3)
    per_vec = 8 if dt == synth.BF16 else 4  # row stride must be a multiple of 16 bytes
    _case(orc, w, seed=vocab, row_stride=-(-vocab // per_vec) * per_vec)


def test_padded_row_stride(orc):
    w = synth.scaled(synth.WORKLOADS["single_seq"], vocab=5000, batch=2)
    _case(orc, w, seed=5, row_stride=5000 + 24)


def test_many_rows_one_slice_each(orc):
    # more rows than resident CTA slots: one CTA per row, several waves
    w = synth.scaled(synth.WORKLOADS["batched"], vocab=3000, batch=40, block=64, seq_len=1024,
                     prompt_len=256, active_block=4)
    _case(orc, w, seed=9)


def test_neg_inf_and_exact_ties(orc):
    nat = native()
    w = synth.scaled(synth.WORKLOADS["tiny"], vocab=777, logits_dtype=synth.BF16, n_unmask=5)
    rng = np.random.default_rng(13)
    st = synth.make_state(rng, w)
    x = rng.standard_normal((w.n_rows, w.vocab)).astype(np.float32)
    x[0, :] = -np.inf
    x[0, 100] = 2.0                     # one-hot: entropy 0, conf 1
    x[1, [5, 300, 600]] = 9.0           # exact three-way tie for the argmax
    x[2, ::2] = -np.inf                 # half the vocabulary banned
    x[3, :] = 0.5                       # uniform: entropy ln V
    x[4, :] = x[5, :]                   # two identical rows: equal confidence, position decides
    logits = synth.f32_to_bf16_bits(x)
    gpu = run_decode_gpu(nat, logits, st, w.n_unmask, w.tau, st.step, row_stride=784)
    ref = run_decode_oracle(orc, logits, st, w.n_unmask, w.tau, st.step)
    check_decode(gpu, ref, st, w.n_unmask, w.tau, st.step)
    assert gpu["token"][0] == 100 and gpu["entropy"][0] == 0.0 and gpu["conf"][0] == 1.0
    assert gpu["token"][1] == 5
    assert abs(gpu["entropy"][3] - np.log(777)) < 1e-4


def test_empty_and_short_sequences(orc):
    nat = native()
    rng = np.random.default_rng(17)
    V, L = 2048, 64
    counts = [0, 3, 0, 9, 1]
    B = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    pos = np.concatenate([np.sort(rng.choice(L, size=c, replace=False)) for c in counts]).astype(np.int32)
    is_masked = np.zeros((B, L), np.uint8)
    for b in range(B):
        is_masked[b, pos[off[b]:off[b + 1]]] = 1
    st = synth.DecodeState(is_masked, rng.integers(0, V, (B, L)).astype(np.int32),
                           np.full((B, L), -1, np.int32), 3, 0, L, pos, off)
    logits = synth.make_logits(rng, int(off[-1]), V, synth.BF16)
    gpu = run_decode_gpu(nat, logits, st, 4, 0.7, 3)
    ref = run_decode_oracle(orc, logits, st, 4, 0.7, 3)
    check_decode(gpu, ref, st, 4, 0.7, 3)
    assert list(gpu["unmask_rows"][0]) == [-1] * 4 and gpu["max_entropy"][0] == -np.inf
    assert gpu["refresh"][0] == 0 and gpu["refresh"][2] == 0
    assert (gpu["unmask_rows"][4] >= 0).sum() == 1


def test_no_rows_at_all(orc):
    nat = native()
    import torch
    B, L = 3, 16
    st = synth.DecodeState(np.zeros((B, L), np.uint8), np.zeros((B, L), np.int32),
                           np.full((B, L), -1, np.int32), 0, 0, L, np.zeros(0, np.int32),
                           np.zeros(B + 1, np.int32))
    gpu = run_decode_gpu(nat, np.zeros((0, 64), np.uint16), st, 2, 0.5, 0)
    assert (gpu["unmask_rows"] == -1).all() and (gpu["refresh"] == 0).all()
    assert np.isneginf(gpu["max_entropy"]).all()


def test_repeated_calls_reuse_the_workspace(orc):
    # counters in the workspace must return to zero after every call
    nat = native()
    w = synth.WORKLOADS["single_seq"]
    rng = np.random.default_rng(23)
    st = synth.make_state(rng, w)
    ws = nat.new_workspace(nat.ec_decode_workspace_size(w.n_rows, w.batch))
    first = None
    for i in range(5):
        logits = synth.make_logits(np.random.default_rng(100 + (i % 2)), w.n_rows, w.vocab,
                                   w.logits_dtype)
        gpu = run_decode_gpu(nat, logits, st, w.n_unmask, w.tau, st.step, workspace=ws)
        if i % 2 == 0:
            if first is None:
                first = gpu
            for k in ("token", "conf", "entropy", "unmask_rows", "refresh"):
                assert np.array_equal(gpu[k], first[k]), k  # deterministic
    ref = run_decode_oracle(orc, synth.make_logits(np.random.default_rng(100), w.n_rows, w.vocab,
                                                   w.logits_dtype), st, w.n_unmask, w.tau, st.step)
    check_decode(first, ref, st, w.n_unmask, w.tau, st.step)


@pytest.mark.parametrize("dt", [synth.BF16, synth.F32])
def test_batched_ragged_vocab(orc, dt):
    # full batched size with an odd vocabulary: rows cut over two or three CTAs,
    # the piece ending each row holding the vocab % 8 (bf16) or % 4 (fp32) tail
    w = synth.scaled(synth.WORKLOADS["batched"], vocab=152063, logits_dtype=dt)
    per_vec = 8 if dt == synth.BF16 else 4
    _case(orc, w, seed=31, row_stride=-(-w.vocab // per_vec) * per_vec)


def test_repeated_calls_split_rows(orc):
    # rows split over several CTAs: the tickets must return to zero after every
    # call and repeated calls give identical results
    nat = native()
    w = synth.WORKLOADS["long_ctx"]
    rng = np.random.default_rng(41)
    st = synth.make_state(rng, w)
    logits = synth.make_logits(rng, w.n_rows, w.vocab, w.logits_dtype, w.near_uniform_frac)
    ws = nat.new_workspace(nat.ec_decode_workspace_size(w.n_rows, w.batch))
    runs = [run_decode_gpu(nat, logits, st, w.n_unmask, w.tau, st.step, workspace=ws)
            for _ in range(4)]
    for gpu in runs[1:]:
        for k in ("token", "conf", "entropy", "unmask_rows", "refresh", "max_entropy"):
            assert np.array_equal(gpu[k], runs[0][k]), k
    ref = run_decode_oracle(orc, logits, st, w.n_unmask, w.tau, st.step)
    check_decode(runs[0], ref, st, w.n_unmask, w.tau, st.step)


@pytest.mark.parametrize("dt", [synth.BF16, synth.F32])
def test_long_rows_with_neg_inf_ties_and_signed_zeros(orc, dt):
    # rows long enough to be split into a head and pool chunks (>= 64 KB): -inf
    # logits anywhere (the bf16 fold's guarded refold), maxima placed in the
    # head, in a pool chunk and in the last elements after the final whole
    # vector, exact ties across pieces, and +0 / -0 maxima
    nat = native()
    V = 70003 if dt == synth.BF16 else 40001
    w = synth.scaled(synth.WORKLOADS["batched"], vocab=V, logits_dtype=dt, batch=2, block=8,
                     seq_len=256, prompt_len=64, active_block=2, n_unmask=3)
    rng = np.random.default_rng(77)
    st = synth.make_state(rng, w)
    x = rng.standard_normal((w.n_rows, V)).astype(np.float32)
    x[0, ::3] = -np.inf                       # a third banned, max in the head
    x[0, 17] = 6.0
    x[1, V - 2] = 7.0                         # max among the last elements
    x[1, 1000:1100] = -np.inf
    x[2, [5, V // 2, V - 900]] = 8.0          # tie: head, middle, pool chunk -> 5
    x[3, :] = -np.inf                         # one-hot at the very end of the row
    x[3, V - 1] = 0.0
    x[4, :] = -1.0                            # -0 before +0: the maximum is 0, first at -0
    x[4, V // 3] = -0.0
    x[4, V - 3] = 0.0
    x[5, V - 5000] = 9.0                      # max in a pool chunk
    x[6, :V // 2] = -np.inf                   # the first half banned
    x[7, :] = 0.25                            # uniform
    logits = synth.f32_to_bf16_bits(x) if dt == synth.BF16 else x
    per_vec = 8 if dt == synth.BF16 else 4
    stride = -(-V // per_vec) * per_vec
    gpu = run_decode_gpu(nat, logits, st, w.n_unmask, w.tau, st.step, row_stride=stride)
    ref = run_decode_oracle(orc, logits, st, w.n_unmask, w.tau, st.step)
    check_decode(gpu, ref, st, w.n_unmask, w.tau, st.step)
    assert gpu["token"][0] == 17 and gpu["token"][1] == V - 2 and gpu["token"][2] == 5
    assert gpu["token"][3] == V - 1 and gpu["entropy"][3] == 0.0
    assert gpu["token"][4] == V // 3 and gpu["token"][5] == V - 5000
    assert abs(gpu["entropy"][7] - np.log(V)) < 1e-4


def test_report_exclusions():
    for name, seed, excl in REPORT:
        if excl:
            print(f"excluded decisions: workload={name} seed={seed} sequences={excl}")
