"""Checkpoint / resume of a GPU trajectory: a trajectory saved after some steps and
resumed in a fresh driver makes the same decisions and ends with bit-identical
state and caches as the run that went on without stopping."""
import os

import numpy as np
import pytest
import torch

from entropy_gated_kv_decode_b300 import synth
from gpu_helpers import host, native

pytestmark = pytest.mark.gpu

SMALL = synth.scaled(synth.WORKLOADS["trajectory"], vocab=3000, seq_len=256, prompt_len=192,
                     block=16, n_heads=2, n_kv_heads=2, head_dim=64, n_layers=2, n_steps=32,
                     tau=2.5)


@pytest.mark.parametrize("policy,ffn", [(("block",), 0), (("sliding", 20), 256)])
def test_resume_is_bit_exact(tmp_path, policy, ffn):
    native()
    from entropy_gated_kv_decode_b300.trajectory import Trajectory
    w = synth.scaled(SMALL, ffn=ffn)
    a = Trajectory(w, seed=7, trace=True, policy=policy)
    a.warm_up()
    a.reset()
    for _ in range(12):
        a.step()
    path = os.path.join(tmp_path, "ckpt.pt")
    a.save(path)
    for _ in range(w.n_steps - 12):
        a.step()
    torch.cuda.synchronize()
    rest_a = a.records[12:]

    b = Trajectory(w, seed=7, trace=True, policy=policy)
    b.warm_up()
    b.load(path)
    for _ in range(w.n_steps - 12):
        b.step()
    torch.cuda.synchronize()
    assert [(r.full, r.rows, r.refresh) for r in b.records] == \
        [(r.full, r.rows, r.refresh) for r in rest_a]
    assert any(not r.full for r in b.records)  # the resumed part has partial forwards
    for name in ("is_masked", "tokens", "decode_step", "k_cache", "v_cache"):
        assert np.array_equal(host(getattr(a, name)), host(getattr(b, name))), name
    with pytest.raises(ValueError):
        Trajectory(w, seed=8, policy=policy).load(path)
