"""Pins of the oracle's per-row decode statistics (entropy, confidence, token)
against facts fixed by the mathematics, not by the oracle's own formula.

EntropyCache (Arabic technical summary, section 2 "Algorithm workflow", the
E_{t+1} equation) defines the per-row entropy -sum_j p_ij log p_ij of the
softmax distribution a token is decoded from; the Italian summary ("Algoritmo
di Funzionamento", step 1) says new tokens are decoded from the logits.
"""
import math

import mpmath
import numpy as np
import pytest

from entropy_gated_kv_decode_b300 import synth

mpmath.mp.dps = 40


def closed_form(row):
    """High-precision H, conf via the log-partition form H = ln Z - sum_j p_j x_j,
    an algebraically different route from the oracle's -sum p ln p."""
    xs = [mpmath.mpf(float(v)) for v in row if not math.isinf(v) or v > 0]
    z = mpmath.fsum(mpmath.e ** x for x in xs)
    mean_x = mpmath.fsum(x * mpmath.e ** x for x in xs) / z
    h = mpmath.log(z) - mean_x
    conf = mpmath.e ** max(xs) / z
    return float(h), float(conf)


@pytest.mark.parametrize("vocab", [1, 4, 1024, 126464, 152064])
@pytest.mark.parametrize("dtype", ["f64", "f32", "bf16"])
def test_uniform_row_has_entropy_ln_v(orc, vocab, dtype):
    row = np.full((2, vocab), 1.5, np.float32)
    row[1] = -3.25
    x = {"f64": row.astype(np.float64), "f32": row, "bf16": synth.f32_to_bf16_bits(row)}[dtype]
    h, c, t = orc.row_stats(x)
    # float64 summation of V equal terms: error at most ~ V * eps * ln V
    bound = vocab * 2.3e-16 * max(math.log(vocab), 1.0) + 1e-15
    assert np.allclose(h, math.log(vocab), rtol=0, atol=bound)
    assert np.allclose(c, 1.0 / vocab, rtol=vocab * 2.3e-16 + 1e-15, atol=0)
    assert list(t) == [0, 0]  # all tied: the lowest index


@pytest.mark.parametrize("hot", [0, 3, 1023])
def test_one_hot_row_has_zero_entropy(orc, hot):
    row = np.full((1, 1024), -np.inf)
    row[0, hot] = 0.75
    h, c, t = orc.row_stats(row)
    assert h[0] == 0.0 and c[0] == 1.0 and t[0] == hot


def test_masked_out_tokens_reduce_to_smaller_uniform(orc):
    # [0, 0, 0, -inf]: uniform over three tokens
    h, c, t = orc.row_stats(np.array([[0.0, 0.0, 0.0, -np.inf]]))
    assert abs(h[0] - math.log(3)) < 1e-14 and abs(c[0] - 1 / 3) < 1e-15 and t[0] == 0


@pytest.mark.parametrize("a", [2.0, 7.5, 15.0, -3.0, 0.125])
@pytest.mark.parametrize("vocab,where", [(4, 0), (4, 2), (1024, 511), (126464, 126463)])
def test_two_level_row_matches_binary_entropy_closed_form(orc, a, vocab, where):
    # one logit a at index `where`, all others 0: p = e^a/(e^a + V - 1) and
    # H = -p ln p - (1-p) ln((1-p)/(V-1)).
    row = np.zeros((1, vocab))
    row[0, where] = a
    h, c, t = orc.row_stats(row)
    ea = mpmath.e ** mpmath.mpf(a)
    p = ea / (ea + vocab - 1)
    hx = -p * mpmath.log(p) - (1 - p) * mpmath.log((1 - p) / (vocab - 1))
    # float64 rounding of a V-term sum: relative error up to ~ V * eps
    rel = vocab * 2.3e-16 + 1e-15
    assert abs(h[0] - float(hx)) < rel * (math.log(vocab) + abs(a) + 1)
    if a > 0:
        assert abs(c[0] - float(p)) < rel * float(p) and t[0] == where
    else:
        first_zero = 1 if where == 0 else 0
        cx = float(1 / (ea + vocab - 1))
        assert abs(c[0] - cx) < rel * cx and t[0] == first_zero


# Four-token rows, every value exact in bf16.
HAND = [
    [0, 0, 0, 0],
    [2, 1, 0, 0],
    [3, 0, 0, 0],
    [1, 1, 0, 0],
    [8, 0, 0, 0],
    [0, 2, 2, -1],
    [-1, -2, -3, -4],
]


@pytest.mark.parametrize("row", HAND)
def test_four_token_hand_examples(orc, row):
    x = np.array([row], np.float64)
    h, c, t = orc.row_stats(x)
    hx, cx = closed_form(row)
    assert abs(h[0] - hx) < 1e-13
    assert abs(c[0] - cx) < 1e-14
    assert t[0] == int(np.argmax(x[0]))  # numpy: first maximal index


def test_hand_examples_worked_by_hand(orc):
    # rows [2,1,0,0], [3,0,0,0], [1,1,0,0], [8,0,0,0] written out by hand:
    # Z = sum e^x, H = ln Z - sum x e^x / Z, conf = e^max / Z
    e = math.e
    cases = [
        (e**2 + e + 2, (2 * e**2 + e), e**2),
        (e**3 + 3, 3 * e**3, e**3),
        (2 * e + 2, 2 * e, e),
        (e**8 + 3, 8 * e**8, e**8),
    ]
    h, c, t = orc.row_stats(np.array([[2, 1, 0, 0], [3, 0, 0, 0], [1, 1, 0, 0], [8, 0, 0, 0]],
                                     np.float64))
    for i, (z, xe, top) in enumerate(cases):
        assert abs(h[i] - (math.log(z) - xe / z)) < 1e-13
        assert abs(c[i] - top / z) < 1e-15
    assert list(t) == [0, 0, 0, 0]


def test_invariances_and_bounds(orc):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((16, 300)) * rng.uniform(0.1, 4, size=(16, 1))
    h, c, t = orc.row_stats(x)
    # bounds 0 <= H <= ln V, conf in (1/V, 1]
    assert np.all(h >= 0) and np.all(h <= math.log(300) + 1e-12)
    assert np.all(c >= 1 / 300) and np.all(c <= 1)
    # shift invariance (a power of two keeps the shifted values exact)
    h2, c2, t2 = orc.row_stats(x + 64.0)
    assert np.allclose(h, h2, atol=1e-11) and np.allclose(c, c2, rtol=1e-11)
    assert np.array_equal(t, t2)
    # permutation invariance of H and conf; the token follows the permutation
    perm = rng.permutation(300)
    h3, c3, t3 = orc.row_stats(x[:, perm])
    assert np.allclose(h, h3, atol=1e-12) and np.allclose(c, c3, rtol=1e-12)
    assert np.array_equal(perm[t3], t)
    # the argmax is numpy's first maximal index
    assert np.array_equal(t, np.argmax(x, axis=1))


def test_two_form_identity_on_random_rows(orc):
    # H = ln S - T/S with S = sum e^{x-m}, T = sum e^{x-m}(x-m) (numpy, float64)
    rng = np.random.default_rng(11)
    x = rng.standard_normal((8, 5000)) * 3
    x[:, 17] += 12
    h, c, _ = orc.row_stats(x)
    d = x - x.max(axis=1, keepdims=True)
    e = np.exp(d)
    s = e.sum(axis=1)
    tt = (e * d).sum(axis=1)
    assert np.allclose(h, np.log(s) - tt / s, rtol=0, atol=1e-10)
    assert np.allclose(c, 1 / s, rtol=1e-12)


def test_temperature_limits(orc):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 64))
    h_cold, c_cold, _ = orc.row_stats(x * 1e4)
    assert np.all(h_cold < 1e-6) and np.all(c_cold > 1 - 1e-6)
    h_hot, _, _ = orc.row_stats(x * 1e-9)
    assert np.allclose(h_hot, math.log(64), atol=1e-12)


def test_ties_pick_lowest_index(orc):
    x = np.zeros((3, 10))
    x[0, [4, 2, 9]] = 5.0
    x[1, [9]] = 1.0
    x[2, [0, 9]] = 2.0
    _, _, t = orc.row_stats(x)
    assert list(t) == [2, 9, 0]


def test_row_stride_is_honoured(orc):
    rng = np.random.default_rng(5)
    wide = rng.standard_normal((5, 40))
    h_full, c_full, t_full = orc.row_stats(np.ascontiguousarray(wide[:, :33]))
    import ctypes
    n = 5
    h = np.empty(n)
    c = np.empty(n)
    t = np.empty(n, np.int32)
    rc = orc.lib().orc_row_stats(wide.ctypes.data_as(ctypes.c_void_p), 2, 40, n, 33,
                                 h.ctypes.data_as(ctypes.c_void_p),
                                 c.ctypes.data_as(ctypes.c_void_p),
                                 t.ctypes.data_as(ctypes.c_void_p))
    assert rc == 0
    assert np.array_equal(h, h_full) and np.array_equal(t, t_full)


@pytest.mark.parametrize("cuts", [[0, 100], [0, 1, 2, 3, 4999], [0, 1250, 2500, 3750]])
def test_piece_states_merge_to_the_row_statistics(orc, cuts):
    # The GPU path folds pieces of a row into states (m, S, T, a) in the log2 domain,
    # S = sum 2^y, T = sum 2^y y, y = (x - m) log2 e, and merges two states by
    # rescaling the one with the smaller maximum by f = 2^d, d = (m_lo - m_hi) log2 e:
    # S = f S_lo + S_hi, T = f (d S_lo + T_lo) + T_hi, keeping the larger maximum
    # (lower index on a tie).  Pin that merge against the oracle's direct
    # statistics: H = ln S - ln2 T / S, conf = 1 / S, token = a.
    rng = np.random.default_rng(len(cuts))
    x = rng.standard_normal((4, 5000)) * 2
    x[1, 3333] += 9
    x[2, [10, 4000]] = 7.5  # a tie across pieces
    h, c, t = orc.row_stats(x)
    l2e = 1 / math.log(2)
    bounds = cuts + [x.shape[1]]
    for i in range(x.shape[0]):
        state = None
        for a, z in zip(bounds[:-1], bounds[1:]):
            piece = x[i, a:z]
            m = piece.max()
            y = (piece - m) * l2e
            s = np.exp2(y).sum()
            tt = (np.exp2(y) * y).sum()
            cur = (m, s, tt, a + int(np.argmax(piece)))
            if state is None:
                state = cur
                continue
            hi, lo = (cur, state) if (cur[0] > state[0] or (cur[0] == state[0] and cur[3] < state[3])) else (state, cur)
            d = (lo[0] - hi[0]) * l2e
            f = 2.0 ** d
            state = (hi[0], f * lo[1] + hi[1], f * (d * lo[1] + lo[2]) + hi[2], hi[3])
        m, s, tt, a = state
        assert math.isclose(math.log(s) - math.log(2) * tt / s, h[i], rel_tol=0, abs_tol=1e-10)
        assert math.isclose(1 / s, c[i], rel_tol=1e-12)
        assert a == t[i]
