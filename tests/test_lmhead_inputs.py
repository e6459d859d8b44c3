"""The LM-head inputs and the oracle composition the fused LM-head step is
checked against (host only).

The exact recipe makes every logit an integer multiple of a power of two far
below 2^24 units, so float32 accumulation in any order gives the float64 result:
the integer product, computed here in int64, pins the oracle's projection on
those inputs, and it is what makes bit-exact tokens a fair demand of the GPU."""
import numpy as np

from entropy_gated_kv_decode_b300 import synth


def _ints(bits, unit):
    v = synth.bf16_bits_to_f32(bits).astype(np.float64) / unit
    assert np.array_equal(v, np.round(v))
    return v.astype(np.int64)


def test_exact_recipe_is_small_integers_times_powers_of_two():
    rng = np.random.default_rng(3)
    for hidden in (64, 256, 4096):
        x, w = synth.make_lmhead(rng, 64, 300, hidden)
        assert np.abs(_ints(w, 2.0 ** -6)).max() <= 3
        xf = synth.bf16_bits_to_f32(x).astype(np.float64)
        for i in range(64):
            nz = np.abs(xf[i][xf[i] != 0])
            unit = 2.0 ** np.floor(np.log2(nz.min()))  # the row's smallest power of two
            k = _ints(x[i], unit)
            assert np.abs(k).max() < 256  # bf16 holds every such integer exactly


def test_oracle_projection_is_the_integer_product_on_exact_inputs(orc):
    rng = np.random.default_rng(5)
    for n, v, h in ((24, 517, 320), (16, 300, 4096)):
        x, w = synth.make_lmhead(rng, n, v, h)
        xi = _ints(x, 2.0 ** -16)          # every hidden value is a multiple of 2^-16
        wi = _ints(w, 2.0 ** -6)
        prod = xi @ wi.T                   # int64, exact
        y = orc.projection(x, w)
        assert np.array_equal(y, prod.astype(np.float64) * 2.0 ** -22)
        # float32 holds every logit and every partial sum: each row's integers in
        # its own unit stay far below 2^24
        for i in range(n):
            xf = synth.bf16_bits_to_f32(x[i]).astype(np.float64)
            unit = 2.0 ** np.floor(np.log2(np.abs(xf[xf != 0]).min()))
            ki = _ints(x[i], unit)
            assert np.abs(ki).astype(np.int64) @ np.abs(wi).max(axis=0) < 2 ** 24
        assert np.array_equal(y.astype(np.float32).astype(np.float64), y)


def test_exact_recipe_spans_peaked_and_flat_rows(orc):
    # rows from near one-hot to near uniform, so the gate sees both sides of tau
    rng = np.random.default_rng(7)
    x, w = synth.make_lmhead(rng, 256, 4096, 512)
    h, c, t = orc.row_stats(orc.projection(x, w))
    assert h.min() < 0.5 and h.max() > 0.9 * np.log(4096)
    assert c.max() < 1.0  # no confidence saturates
    assert np.all((t >= 0) & (t < 4096))


def test_lmhead_oracle_composition_equals_decode_on_materialised_logits(orc):
    # the fused step's oracle is projection -> row statistics -> unmask and gate,
    # i.e. the decode step's oracle on the float64 logits
    rng = np.random.default_rng(9)
    wl = synth.scaled(synth.WORKLOADS["tiny"], vocab=700, logits_dtype=synth.BF16)
    st = synth.make_state(rng, wl)
    x, w = synth.make_lmhead(rng, wl.n_rows, wl.vocab, 128)
    logits = orc.projection(x, w)
    h, c, t = orc.row_stats(logits)
    h32, c32, t32 = orc.row_stats(logits.astype(np.float32))  # exact: same values
    assert np.array_equal(t, t32) and np.array_equal(h, h32) and np.array_equal(c, c32)
    g = orc.unmask_gate(c, h, t, st.seq_row_offsets, st.row_pos, wl.seq_len, wl.n_unmask, wl.tau,
                        st.step, st.is_masked, st.tokens, st.decode_step)
    assert (g["unmask_rows"] >= 0).sum() == min(wl.n_unmask, wl.n_rows)
