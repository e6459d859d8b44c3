"""The allocation-free decode entry point (ec_decode_step_noalloc), called
through the C ABI, gives the same results as ec_decode_step with a caller
workspace, on two calls in a row.

It exists for callers that cannot allocate device memory themselves (device
memory owned by a host framework or a fixed pool, or a decode loop where a
cudaMalloc is not acceptable).  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from entropy_gated_kv_decode_b300 import synth
from gpu_helpers import ENTROPY_ATOL, dev, host, native

pytestmark = pytest.mark.gpu

FIELDS = ("token", "conf", "entropy", "unmask_rows", "max_entropy", "refresh",
          "is_masked", "tokens", "decode_step")


def _buffers(w, st):
    B, N, n = w.batch, w.n_rows, w.n_unmask
    cuda = torch.device("cuda")
    return dict(token=torch.full((N,), -5, dtype=torch.int32, device=cuda),
                conf=torch.full((N,), float("nan"), device=cuda),
                entropy=torch.full((N,), float("nan"), device=cuda),
                unmask_rows=torch.full((B * n,), -5, dtype=torch.int32, device=cuda),
                max_entropy=torch.full((B,), float("nan"), device=cuda),
                refresh=torch.full((B,), 9, dtype=torch.uint8, device=cuda),
                is_masked=dev(st.is_masked.copy()), tokens=dev(st.tokens.copy()),
                decode_step=dev(st.decode_step.copy()))


def _args(w, st, logits, o):
    return (logits, dev(st.seq_row_offsets), dev(st.row_pos), w.seq_len, w.n_unmask, w.tau,
            st.step, o["token"], o["conf"], o["entropy"], o["unmask_rows"], o["max_entropy"],
            o["refresh"], o["is_masked"], o["tokens"], o["decode_step"])


def _compare_one_call(nat, w, seed, tag):
    st = synth.make_state(np.random.default_rng(0), w)
    rng = np.random.default_rng(seed)
    logits = dev(synth.make_logits(rng, w.n_rows, w.vocab, w.logits_dtype, w.near_uniform_frac))
    ref = _buffers(w, st)
    ws = nat.new_workspace(nat.ec_decode_workspace_size(w.n_rows, w.batch))
    nat.ec_decode_step(*_args(w, st, logits, ref), ws)
    got = _buffers(w, st)
    nat.ec_decode_step_noalloc(*_args(w, st, logits, got))
    torch.cuda.synchronize()
    for k in FIELDS:
        a, b = host(ref[k]), host(got[k])
        if k in ("conf", "entropy", "max_entropy"):
            assert np.allclose(a, b, rtol=1e-6, atol=ENTROPY_ATOL, equal_nan=False), (tag, k)
        else:
            assert np.array_equal(a, b), (tag, k)


@pytest.mark.parametrize("name", ["single_seq", "batched"])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(name):
    nat = native()
    w = synth.WORKLOADS[name]
    for call in range(2):  # the second call must not see the first call's leftovers
        _compare_one_call(nat, w, 100 + call, call)


def test_noalloc_alternating_shapes():
    # the scratch layout moves with n_rows and batch: a call after a larger or a
    # smaller one must still start from cleared counters
    nat = native()
    for i, name in enumerate(["batched", "single_seq", "tiny", "batched", "single_seq"]):
        _compare_one_call(nat, synth.WORKLOADS[name], 200 + i, (i, name))


def test_noalloc_rejects_requests_beyond_its_scratch():
    nat = native()
    n_rows = 4096  # needs more than the 2 MiB built-in scratch
    lib = nat.lib()
    assert nat.ec_decode_workspace_size(n_rows, 1) > 2 << 20
    rc = lib.ec_decode_step_noalloc(0x1000, 1, 1024, n_rows, 1024, 0x2000, 0x3000, 1, 8192, 2,
                                    0.5, 0, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000, 0x9000,
                                    0xa000, 0xb000, 0xc000, None)
    assert rc == -8
    assert "scratch" in nat.status_str(rc)


def test_noalloc_status_reports_a_timeout_and_clears():
    # the allocation-free call's device status: clean after a normal call,
    # EC_DEV_TIMEOUT after a call whose waits were made to run out, clean again
    # after the next normal call
    nat = native()
    w = synth.scaled(synth.WORKLOADS["batched"], batch=4, block=16, seq_len=512, prompt_len=128,
                     active_block=2, vocab=20000)
    st = synth.make_state(np.random.default_rng(0), w)
    logits = dev(synth.make_logits(np.random.default_rng(3), w.n_rows, w.vocab, w.logits_dtype))
    nat.ec_decode_step_noalloc(*_args(w, st, logits, _buffers(w, st)))
    assert nat.ec_decode_noalloc_read_status() == 0
    nat.ec_debug_set_wait_limit(300)
    try:
        nat.ec_decode_step_noalloc(*_args(w, st, logits, _buffers(w, st)))
        bits = nat.ec_decode_noalloc_read_status()
    finally:
        nat.ec_debug_set_wait_limit(0)
    assert bits & nat.DEV_TIMEOUT, f"status {bits:#x}"
    _compare_one_call(nat, w, 3, "after timeout")
    assert nat.ec_decode_noalloc_read_status() == 0
