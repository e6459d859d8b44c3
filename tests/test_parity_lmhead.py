"""GPU LM-head fused decode-and-gate step (ec_lmhead_decode_step) against the
float64 oracle composition: projection, then the row statistics, then the
unmasking and the gate — the decode step's oracle on the logits that the fused
kernel never writes out.

On the exact-integer inputs every float32 logit equals the float64 one, so the
tokens must match bit for bit and the rest to the decode step's tolerances; on
Gaussian inputs rows whose two largest logits are closer than the float32
accumulation bound are excluded from the token check and reported."""
import math

import numpy as np
import pytest
import torch

from entropy_gated_kv_decode_b300 import synth
from gpu_helpers import (CONF_RTOL, ENTROPY_ATOL, check_decode, dev, host, native,
                         run_decode_oracle)

pytestmark = pytest.mark.gpu

HIDDEN = 4096
REPORT = []


def run_lmhead_gpu(nat, x, w, state, n_unmask, tau, step, workspace=None):
    n_rows = x.shape[0]
    B, L = state.is_masked.shape
    cuda = torch.device("cuda")
    out = dict(
        token=torch.full((n_rows,), -7, dtype=torch.int32, device=cuda),
        conf=torch.full((n_rows,), float("nan"), device=cuda),
        entropy=torch.full((n_rows,), float("nan"), device=cuda),
        unmask_rows=torch.full((B * n_unmask,), -7, dtype=torch.int32, device=cuda),
        max_entropy=torch.full((B,), float("nan"), device=cuda),
        refresh=torch.full((B,), 7, dtype=torch.uint8, device=cuda),
    )
    im, tk, ds = dev(state.is_masked.copy()), dev(state.tokens.copy()), dev(state.decode_step.copy())
    ws = workspace if workspace is not None else nat.new_workspace(
        nat.ec_lmhead_workspace_size(n_rows, w.shape[0], B))
    nat.ec_lmhead_decode_step(dev(x), dev(w), dev(state.seq_row_offsets), dev(state.row_pos), L,
                              n_unmask, tau, step, out["token"], out["conf"], out["entropy"],
                              out["unmask_rows"], out["max_entropy"], out["refresh"], im, tk, ds, ws)
    bits = nat.ec_read_device_status(ws)
    res = {k: host(v) for k, v in out.items()}
    res["unmask_rows"] = res["unmask_rows"].reshape(B, n_unmask)
    res.update(is_masked=host(im), tokens=host(tk), decode_step=host(ds), status=bits)
    return res


def _exact_case(orc, w, hidden=HIDDEN, seed=0):
    nat = native()
    rng = np.random.default_rng(seed)
    st = synth.make_state(rng, w)
    x, wl = synth.make_lmhead(rng, w.n_rows, w.vocab, hidden)
    gpu = run_lmhead_gpu(nat, x, wl, st, w.n_unmask, w.tau, st.step)
    ref = run_decode_oracle(orc, orc.projection(x, wl), st, w.n_unmask, w.tau, st.step)
    excluded = check_decode(gpu, ref, st, w.n_unmask, w.tau, st.step)
    REPORT.append((w.name, w.vocab, hidden, seed, sorted(excluded)))
    assert len(excluded) <= max(1, w.batch // 4), f"too many excluded decisions: {excluded}"
    return gpu


@pytest.mark.parametrize("name", ["single_seq", "batched", "long_ctx"])
def test_workloads_full_size_exact(orc, name):
    _exact_case(orc, synth.WORKLOADS[name])


@pytest.mark.parametrize("vocab,hidden", [(1, 64), (255, 128), (257, 64), (1000, 192),
                                          (70001, 256)])
def test_ragged_vocab_and_hidden(orc, vocab, hidden):
    # a single column, one column past a tile, partial last tiles, K of 1-4 steps
    w = synth.scaled(synth.WORKLOADS["single_seq"], vocab=vocab, batch=3, seq_len=256,
                     prompt_len=64, block=45, active_block=2, n_unmask=3)
    _exact_case(orc, w, hidden=hidden, seed=vocab)


def test_ragged_rows_over_many_row_tiles(orc):
    # 37 sequences of 37 rows: 1369 rows, 11 row tiles, the last one ragged
    w = synth.scaled(synth.WORKLOADS["batched"], vocab=3000, batch=37, block=37, seq_len=512,
                     prompt_len=128, active_block=3)
    _exact_case(orc, w, hidden=128, seed=11)


def test_one_row_tile_per_sm(orc):
    # the largest row count: 128 rows per SM, one CTA per row tile
    nat = native()
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    w = synth.scaled(synth.WORKLOADS["batched"], vocab=600, batch=n_sm, block=128, seq_len=256,
                     prompt_len=0, active_block=1)
    assert w.n_rows == 128 * n_sm
    _exact_case(orc, w, hidden=64, seed=13)
    # one row more is refused before anything runs
    n = w.n_rows + 1
    cuda = torch.device("cuda")
    i32 = lambda k: torch.zeros(k, dtype=torch.int32, device=cuda)
    f32 = lambda k: torch.zeros(k, dtype=torch.float32, device=cuda)
    u8 = lambda k: torch.zeros(k, dtype=torch.uint8, device=cuda)
    with pytest.raises(nat.ECError, match="SHAPE"):
        nat.ec_lmhead_decode_step(
            torch.zeros((n, 64), dtype=torch.bfloat16, device=cuda),
            torch.zeros((600, 64), dtype=torch.bfloat16, device=cuda),
            torch.tensor([0, n], dtype=torch.int32, device=cuda), i32(n), n, 1, 0.5, 0,
            i32(n), f32(n), f32(n), i32(1), f32(1), u8(1), u8(n), i32(n), i32(n),
            nat.new_workspace(nat.ec_lmhead_workspace_size(n, 600, 1)))


def test_gaussian_inputs_with_accumulation_bound(orc):
    nat = native()
    w = synth.scaled(synth.WORKLOADS["batched"], vocab=20000, batch=4, block=64)
    rng = np.random.default_rng(17)
    st = synth.make_state(rng, w)
    hidden = 1024
    x, wl = synth.make_lmhead(rng, w.n_rows, w.vocab, hidden, exact=False)
    gpu = run_lmhead_gpu(nat, x, wl, st, w.n_unmask, w.tau, st.step)
    assert gpu["status"] == 0
    logits = orc.projection(x, wl)
    h, c, t = orc.row_stats(logits)
    # float32 accumulation of `hidden` products (truncation or rounding):
    # |error| <= hidden * 2^-23 * sum_e |x_e w_je|
    ax = synth.f32_to_bf16_bits(np.abs(synth.bf16_bits_to_f32(x)))
    aw = synth.f32_to_bf16_bits(np.abs(synth.bf16_bits_to_f32(wl)))
    bound = hidden * 2.0 ** -23 * orc.projection(ax, aw).max(axis=1)
    top2 = -np.partition(-logits, 1, axis=1)[:, :2]
    near = np.nonzero(top2[:, 0] - top2[:, 1] <= 2 * bound)[0]
    far = np.setdiff1d(np.arange(w.n_rows), near)
    REPORT.append(("gauss", w.vocab, hidden, 17, near.tolist()))
    assert len(near) <= w.n_rows // 20
    assert np.array_equal(gpu["token"][far], t[far])
    # entropy moves by at most 2 * bound per row (each logit off by <= bound)
    assert np.all(np.abs(gpu["entropy"] - h) <= ENTROPY_ATOL + 2 * bound)
    assert np.all(np.abs(gpu["conf"] - c) <= CONF_RTOL * c + 2 * bound * c + 1e-7)
    # the gate is consistent with the kernel's own per-row outputs
    for b in range(w.batch):
        rows = np.arange(st.seq_row_offsets[b], st.seq_row_offsets[b + 1])
        own = sorted(rows.tolist(), key=lambda r: (-gpu["conf"][r], st.row_pos[r]))[:w.n_unmask]
        assert list(gpu["unmask_rows"][b]) == own
        e = max(gpu["entropy"][r] for r in own)
        assert gpu["max_entropy"][b] == np.float32(e)
        assert gpu["refresh"][b] == (1 if e > np.float32(w.tau) else 0)


def test_no_rows(orc):
    nat = native()
    B, L = 3, 16
    st = synth.DecodeState(np.zeros((B, L), np.uint8), np.zeros((B, L), np.int32),
                           np.full((B, L), -1, np.int32), 0, 0, L, np.zeros(0, np.int32),
                           np.zeros(B + 1, np.int32))
    _, wl = synth.make_lmhead(np.random.default_rng(2), 1, 512, 64)
    gpu = run_lmhead_gpu(nat, np.zeros((0, 64), np.uint16), wl, st, 2, 0.5, 0)
    assert gpu["status"] == 0
    assert (gpu["unmask_rows"] == -1).all() and (gpu["refresh"] == 0).all()
    assert np.isneginf(gpu["max_entropy"]).all()


def test_repeated_calls_reuse_the_workspace(orc):
    nat = native()
    w = synth.scaled(synth.WORKLOADS["batched"], vocab=9000)
    rng = np.random.default_rng(19)
    st = synth.make_state(rng, w)
    x, wl = synth.make_lmhead(rng, w.n_rows, w.vocab, 256)
    ws = nat.new_workspace(nat.ec_lmhead_workspace_size(w.n_rows, w.vocab, w.batch))
    runs = [run_lmhead_gpu(nat, x, wl, st, w.n_unmask, w.tau, st.step, workspace=ws)
            for _ in range(3)]
    for gpu in runs[1:]:
        for k in ("token", "conf", "entropy", "unmask_rows", "refresh", "max_entropy"):
            assert np.array_equal(gpu[k], runs[0][k]), k
    ref = run_decode_oracle(orc, orc.projection(x, wl), st, w.n_unmask, w.tau, st.step)
    check_decode(runs[0], ref, st, w.n_unmask, w.tau, st.step)


def test_report_exclusions():
    for name, vocab, hidden, seed, excl in REPORT:
        if excl:
            print(f"excluded: case={name} vocab={vocab} hidden={hidden} seed={seed} -> {excl}")
