"""GPU seed score (ec_cover_seed_score) against the float64 oracle on the same
seeded inputs: d_in, d_out and the score of every candidate row within the
bounds of tests/cover_score_check.py, rows that are not candidates left
unchanged, the seeds exactly the ranking of the GPU's own scores and the
oracle's up to near ties.  Every candidate row is compared, at full size too."""
import numpy as np
import pytest
import torch

import cover_score_check as chk
from gpu_helpers import dev, host, native

pytestmark = pytest.mark.gpu


def run_gpu(case, n_seed):
    nat = native()
    q, kc, idx, cnt, role, drafted, u, scale = case
    B, R = role.shape
    L, H = kc.shape[1], q.shape[2]
    outs = [torch.full((B, R), chk.CANARY, dtype=torch.float32, device="cuda") for _ in range(3)]
    seeds = torch.full((B, n_seed), -7, dtype=torch.int32, device="cuda") if n_seed else None
    ws = nat.new_workspace(nat.ec_cover_score_workspace_size(B, L, R, H))
    nat.ec_cover_seed_score(dev(q), dev(kc), dev(idx), dev(cnt), dev(role), dev(drafted), dev(u),
                            scale, n_seed, outs[0], outs[1], outs[2], seeds, ws)
    status = nat.ec_read_device_status(ws)
    got = [host(t) for t in outs]
    got.append(host(seeds) if n_seed else np.zeros((B, 0), np.int32))
    return got, status


def compare(orc, case, n_seed):
    q, kc, idx, cnt, role, drafted, u, scale = case
    got, status = run_gpu(case, n_seed)
    ref = orc.cover_seed_score(q, kc, idx, cnt, role, drafted, u, scale, n_seed)
    chk.check(got, ref, idx, cnt, role, n_seed)
    return got, status


@pytest.mark.parametrize("name,n_drafted,n_seed,std", [
    ("single_seq", 2, 4, None), ("batched", 4, 8, None), ("batched", 4, 8, 1.0),
    ("long_ctx", 8, 16, None)])
def test_workloads(orc, name, n_drafted, n_seed, std):
    case = chk.workload_case(orc, name, n_drafted, std)
    assert compare(orc, case, n_seed)[1] == 0


@pytest.mark.parametrize("B,L,R,H,Hkv,D,n_seed", [
    (2, 1, 1, 4, 4, 64, 2),
    (3, 129, 40, 8, 2, 128, 5),
    (2, 300, 77, 7, 1, 64, 100),
    (1, 4100, 20, 2, 1, 128, 0),
    (5, 2049, 130, 14, 2, 128, 9),
])
def test_ragged(orc, B, L, R, H, Hkv, D, n_seed):
    case = chk.ragged_case(np.random.default_rng(L + R), B, L, R, H, Hkv, D)
    assert compare(orc, case, n_seed)[1] == 0


def test_equal_scores_go_to_the_lower_position(orc):
    rng = np.random.default_rng(3)
    q, kc, idx, cnt, role, drafted, u, scale = chk.ragged_case(rng, 2, 90, 30, 4, 2, 64)
    q[:] = 0
    u[:] = 1.25
    got, status = compare(orc, (q, kc, idx, cnt, role, drafted, u, scale), 6)
    assert status == 0
    for b in range(2):
        cand = [int(idx[b, r]) for r in range(cnt[b]) if role[b, r] & 2]
        assert got[3][b].tolist() == (sorted(cand) + [-1] * 6)[:6]


def test_bad_index_drops_the_row(orc):
    nat = native()
    rng = np.random.default_rng(4)
    q, kc, _, cnt, role, drafted, u, scale = chk.ragged_case(rng, 2, 200, 30, 4, 2, 128)
    cnt[:] = 30
    from entropy_gated_kv_decode_b300 import synth
    idx = synth.random_index_set(rng, 2, 200, cnt, stride=33)
    role[0, :6] = [1, 1, 2, 3, 2, 1]
    idx[0, 3] = 200
    got, status = run_gpu((q, kc, idx, cnt, role, drafted, u, scale), 4)
    assert status == nat.DEV_BAD_INDEX
    role_ref, idx_ref = role.copy(), idx.copy()
    role_ref[0, 3], idx_ref[0, 3] = 0, 0
    ref = orc.cover_seed_score(q, kc, idx_ref, cnt, role_ref, drafted, u, scale, 4)
    chk.check(got, ref, idx_ref, cnt, role_ref, 4)


def test_repeated_calls_give_the_same_bits(orc):
    case = chk.workload_case(orc, "single_seq", 2, None, seed=9)
    a, _ = run_gpu(case, 4)
    b, _ = run_gpu(case, 4)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
