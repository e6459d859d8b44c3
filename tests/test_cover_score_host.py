"""The seed-score kernels' per-item code (csrc/cover_score.cuh), compiled for the
host and run item by item in launch order (tests/cover_score_host.cpp), against
the float64 oracle.  It checks the kernels' index arithmetic, key ranges,
merges and ranking without a GPU; the GPU parity test runs the same cases
through the library.  Bounds: tests/cover_score_check.py."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import cover_score_check as chk
from entropy_gated_kv_decode_b300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def host_lib(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    out = str(tmp_path_factory.mktemp("cover_host") / "libcover_host.so")
    subprocess.check_call([cxx, "-O2", "-std=c++17", "-fPIC", "-shared", "-fno-fast-math",
                           "-ffp-contract=off", "-I", os.path.join(ROOT, "include"),
                           "-I", os.path.join(ROOT, "entropy_gated_kv_decode_b300", "csrc"),
                           os.path.join(HERE, "cover_score_host.cpp"), "-o", out])
    lib = ctypes.CDLL(out)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.cover_score_on_host.argtypes = [vp, vp, vp, i64, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                        i32, ctypes.c_float, i32, vp, vp, vp, vp, vp]
    lib.cover_score_on_host.restype = ctypes.c_int
    return lib


def run_host(lib, q, kc, idx, cnt, role, drafted, u, scale, n_seed):
    B, R, H, D = q.shape
    L, Hkv = kc.shape[1], kc.shape[2]
    outs = [np.full((B, R), chk.CANARY, np.float32) for _ in range(3)]
    seeds = np.full((B, max(n_seed, 1)), -7, np.int32)
    status = np.zeros(1, np.uint32)
    arrs = [np.ascontiguousarray(a) for a in (q, kc)]
    ix = np.ascontiguousarray(idx, np.int32)
    cn = np.ascontiguousarray(cnt, np.int32)
    rl = np.ascontiguousarray(role, np.uint8)
    dr = np.ascontiguousarray(drafted, np.uint8)
    uu = np.ascontiguousarray(u, np.float32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    n_chunks = lib.cover_score_on_host(p(arrs[0]), p(arrs[1]), p(ix), ix.shape[1], p(cn), p(rl),
                                       p(dr), p(uu), B, L, R, H, Hkv, D, float(scale), n_seed,
                                       p(outs[0]), p(outs[1]), p(outs[2]), p(seeds), p(status))
    assert n_chunks >= 1
    return outs[0], outs[1], outs[2], seeds[:, :n_seed], int(status[0])


def compare(orc, lib, case, n_seed):
    q, kc, idx, cnt, role, drafted, u, scale = case
    got = run_host(lib, q, kc, idx, cnt, role, drafted, u, scale, n_seed)
    ref = orc.cover_seed_score(q, kc, idx, cnt, role, drafted, u, scale, n_seed)
    chk.check(got[:4], ref, idx, cnt, role, n_seed)
    return got


@pytest.mark.parametrize("name,std", [("batched", None), ("single_seq", 1.0)])
def test_workloads(orc, host_lib, name, std):
    # std 1: sharp attention rows (scores of several units), the rest as generated
    case = chk.workload_case(orc, name, n_drafted=4, std=std)
    assert compare(orc, host_lib, case, n_seed=8)[4] == 0


@pytest.mark.parametrize("B,L,R,H,Hkv,D,n_seed", [
    (2, 1, 1, 4, 4, 64, 2),        # one key
    (3, 129, 40, 8, 2, 128, 5),    # two key ranges, GQA, a ragged tail
    (2, 300, 77, 7, 1, 64, 100),   # more seed slots than candidates
    (1, 4100, 20, 2, 1, 128, 0),   # many key ranges, no seeds asked
])
def test_ragged(orc, host_lib, B, L, R, H, Hkv, D, n_seed):
    case = chk.ragged_case(np.random.default_rng(L + R), B, L, R, H, Hkv, D)
    assert compare(orc, host_lib, case, n_seed)[4] == 0


def test_equal_scores_go_to_the_lower_position(orc, host_lib):
    # q = 0: uniform attention, every candidate has the same d_in and d_out, so
    # equal u gives exactly equal float32 scores
    rng = np.random.default_rng(3)
    q, kc, idx, cnt, role, drafted, u, scale = chk.ragged_case(rng, 2, 90, 30, 4, 2, 64)
    q[:] = 0
    u[:] = 1.25
    got = compare(orc, host_lib, (q, kc, idx, cnt, role, drafted, u, scale), n_seed=6)
    for b in range(2):
        cand = [int(idx[b, r]) for r in range(cnt[b]) if role[b, r] & 2]
        assert got[3][b].tolist() == (sorted(cand) + [-1] * 6)[:6]


def test_bad_index_drops_the_row(orc, host_lib):
    rng = np.random.default_rng(4)
    q, kc, _, cnt, role, drafted, u, scale = chk.ragged_case(rng, 2, 200, 30, 4, 2, 128)
    cnt[:] = 30
    idx = synth.random_index_set(rng, 2, 200, cnt, stride=33)
    role[0, :6] = [1, 1, 2, 3, 2, 1]
    idx[0, 3] = 200  # past the end: the row is dropped
    got = run_host(host_lib, q, kc, idx, cnt, role, drafted, u, scale, 4)
    assert got[4] == 0x8  # EC_DEV_BAD_INDEX
    role_ref, idx_ref = role.copy(), idx.copy()
    role_ref[0, 3], idx_ref[0, 3] = 0, 0  # the oracle with that row taking no part
    ref = orc.cover_seed_score(q, kc, idx_ref, cnt, role_ref, drafted, u, scale, 4)
    chk.check(got[:4], ref, idx_ref, cnt, role_ref, 4)
