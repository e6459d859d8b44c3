"""Seeded synthetic inputs for the EntropyCache decode-and-gate step and the
selective-recompute attention.

This module only draws random numbers and lays them out in the shapes the
library takes.  It holds none of the method's arithmetic: no softmax, entropy,
ranking, gate or index-set logic lives here.  The CUDA path (through the
binding) and the CPU oracle both consume exactly the arrays built here, so the
two sides see bit-identical inputs.

Recipe (one seeded ``numpy.random.Generator`` per call, PCG64):

* Logits.  Spiked rows: ``x = z * T`` with ``z ~ N(0, 1)`` and ``T``
  log-uniform in [0.1, 3], plus ``s ~ U[0, 15]`` added to one uniformly chosen
  token.  Near-uniform rows (a fixed fraction, chosen by a seeded permutation):
  ``x = z / T`` with ``T`` log-uniform in [5, 20], no spike.  bf16 logits are the
  round-to-nearest-even bf16 of the float32 draw.
* Decode state.  Positions ``[0, prompt)`` are prompt (unmasked, never decoded).
  The generated region is split into blocks of ``block`` positions decoded one
  after the other; every block before the active one is fully decoded, in a
  seeded random order, ``n_unmask`` tokens per denoising step.  The active block
  and everything after it is masked (token id = vocab, the [MASK] id).
* LM-head operands (hidden states ``[N, hidden]`` and W_lm ``[V, hidden]``,
  bf16).  The "exact" recipe uses small integers times powers of two, so every
  logit is exactly representable and every float32 partial sum is exact in any
  order: ``W_lm = 2^-6 * U{-3..3}``; hidden row i is
  ``U{-3..3} * 2^a_i + spike_i * 2^b_i``, where ``spike_i`` is the integer
  pattern of W_lm row ``t_i`` on ``m = max(1, hidden / 8)`` random coordinates.
  ``a_i`` sets the spread of the row's logits, about
  ``sigma_i = 4 sqrt(hidden) 2^(a_i - 6)``, to 1/8, 1/4, 1/2 or 1; ``b_i`` sets
  the spike's size, about ``4 m 2^(b_i - 6)``, to 0 (no spike), 2, 4, 8 or 16
  with probabilities .5, .15, .15, .15, .05 (exponents rounded, and
  |a_i - b_i| <= 5 so that every hidden value stays a bf16 integer multiple).
  The "gauss" recipe: hidden ``N(0, 1)``, W_lm ``N(0, (2 / sqrt(hidden))^2)``.
* Attention operands.  Q, the pre-step K/V caches and the freshly projected
  K/V rows are i.i.d. ``N(0, std^2)``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# dtype codes shared by the C ABI and the oracle's typed loaders.
F32 = 0
BF16 = 1
F64 = 2


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic configuration of the decode step and its attention."""

    name: str
    batch: int
    seq_len: int
    prompt_len: int
    block: int
    active_block: int
    vocab: int
    logits_dtype: int
    near_uniform_frac: float
    n_unmask: int
    k: int
    tau: float
    n_heads: int
    n_kv_heads: int
    head_dim: int
    attn_dtype: int
    qkv_std: float
    n_layers: int = 0
    n_steps: int = 0
    ffn: int = 0            # > 0: pre-norm layers with a SwiGLU MLP of this width
    rope_theta: float = 500000.0
    norm_eps: float = 1e-5

    @property
    def rows_per_seq(self) -> int:
        return self.block

    @property
    def n_rows(self) -> int:
        return self.batch * self.block

    @property
    def r_max(self) -> int:
        """Recompute rows per sequence before this step's unmasking: the
        masked block plus the k most recently decoded positions."""
        decoded = self.active_block * self.block
        return self.block + min(self.k, decoded)


_INV_SQRT_128 = 1.0 / math.sqrt(128.0)

WORKLOADS = {
    # N=32 masked rows, V=1024 fp32 logits; attention L=64, H=2, d=64 fp32 N(0,1).
    "tiny": Workload("tiny", batch=1, seq_len=64, prompt_len=0, block=32, active_block=1,
                     vocab=1024, logits_dtype=F32, near_uniform_frac=0.0, n_unmask=4, k=4,
                     tau=1.0, n_heads=2, n_kv_heads=2, head_dim=64, attn_dtype=F32,
                     qkv_std=1.0),
    # One sequence, L=1024 (512 prompt + 512 generated, block 32), V=126464 bf16;
    # attention 48 rows x 1024 keys, H=32, d=128, N(0, 1/sqrt(d)).
    "single_seq": Workload("single_seq", batch=1, seq_len=1024, prompt_len=512, block=32,
                           active_block=8, vocab=126464, logits_dtype=BF16,
                           near_uniform_frac=0.0, n_unmask=2, k=16, tau=0.5, n_heads=32,
                           n_kv_heads=32, head_dim=128, attn_dtype=BF16,
                           qkv_std=_INV_SQRT_128),
    # 8 sequences, L=2048, 64 masked each (512 rows), V=152064 bf16, 30% near-uniform;
    # attention GQA 28/4 heads, d=128, 96 rows per sequence.
    "batched": Workload("batched", batch=8, seq_len=2048, prompt_len=1024, block=64,
                        active_block=8, vocab=152064, logits_dtype=BF16,
                        near_uniform_frac=0.3, n_unmask=4, k=32, tau=0.8, n_heads=28,
                        n_kv_heads=4, head_dim=128, attn_dtype=BF16,
                        qkv_std=_INV_SQRT_128),
    # One sequence, L=8192, 256 masked, V=126464 bf16; attention 288 rows x 8192 keys.
    "long_ctx": Workload("long_ctx", batch=1, seq_len=8192, prompt_len=4096, block=256,
                         active_block=8, vocab=126464, logits_dtype=BF16,
                         near_uniform_frac=0.0, n_unmask=8, k=32, tau=0.5, n_heads=32,
                         n_kv_heads=32, head_dim=128, attn_dtype=BF16,
                         qkv_std=_INV_SQRT_128),
    # 128 denoising steps on L=1024 (768 prompt + 256 generated in blocks of 32),
    # 2 tokens per step, 32 synthetic layers, V=126464 bf16.
    "trajectory": Workload("trajectory", batch=1, seq_len=1024, prompt_len=768, block=32,
                           active_block=0, vocab=126464, logits_dtype=BF16,
                           near_uniform_frac=0.0, n_unmask=2, k=16, tau=0.6, n_heads=32,
                           n_kv_heads=32, head_dim=128, attn_dtype=BF16,
                           qkv_std=_INV_SQRT_128, n_layers=32, n_steps=128),
}


# SimSD verification under its temporal causal mask: 32 sequences, each a
# 1024-token prompt followed by a data section and a mask section of B = 8
# positions (L = 1040); the 16 data and mask positions are the recomputed query
# rows; GQA 32/8 heads, d = 128, bf16 N(0, 1/sqrt(d)).  The decode fields are
# unused.
SIMSD = Workload("simsd", batch=32, seq_len=1040, prompt_len=1024, block=8, active_block=0,
                 vocab=151936, logits_dtype=BF16, near_uniform_frac=0.0, n_unmask=1, k=0,
                 tau=0.5, n_heads=32, n_kv_heads=8, head_dim=128, attn_dtype=BF16,
                 qkv_std=_INV_SQRT_128)


def make_simsd_layout(rng: np.random.Generator, batch: int, prompt_len: int,
                      blk: int) -> tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """SimSD's input layout: ``(section, tau, idx, count)``.  Each sequence is a
    prompt of ``prompt_len`` positions (section 0), a data section and a mask
    section of ``blk`` positions each (sections 1 and 2); one random step map (a
    permutation of 1..blk) per sequence labels both the k-th data position and the
    k-th mask slot.  The query rows are the ``2 blk`` data and mask positions."""
    L = prompt_len + 2 * blk
    section = np.zeros((batch, L), np.uint8)
    tau = np.zeros((batch, L), np.int32)
    for b in range(batch):
        mu = (rng.permutation(blk) + 1).astype(np.int32)
        section[b, prompt_len:prompt_len + blk] = 1
        section[b, prompt_len + blk:] = 2
        tau[b, prompt_len:prompt_len + blk] = mu
        tau[b, prompt_len + blk:] = mu
    idx = np.tile(np.arange(prompt_len, L, dtype=np.int32), (batch, 1))
    count = np.full(batch, 2 * blk, np.int32)
    return section, tau, idx, count


def cover_seeds(rng: np.random.Generator, is_masked: np.ndarray, idx: np.ndarray,
                count: np.ndarray, r_max: int, n_seeds: int) -> np.ndarray:
    """COVER's seed flags ``[batch, r_max]`` uint8: per sequence, ``n_seeds`` rows
    (fewer if there are not enough) drawn at random among the recomputed rows whose
    positions are already decoded (not masked), the tokens a verification pass
    checks."""
    seed = np.zeros((idx.shape[0], r_max), np.uint8)
    for b in range(idx.shape[0]):
        rows = [r for r in range(int(count[b])) if not is_masked[b, idx[b, r]]]
        if rows:
            pick = rng.choice(rows, size=min(n_seeds, len(rows)), replace=False)
            seed[b, pick] = 1
    return seed


def cover_score_inputs(rng: np.random.Generator, is_masked: np.ndarray, idx: np.ndarray,
                       count: np.ndarray, r_max: int, n_drafted: int):
    """Flags and entropies for COVER's seed score: per sequence, ``n_drafted`` of
    the recomputed masked rows are drafted at this step (``drafted`` [batch,
    seq_len] uint8 at their positions); the other masked rows stay masked (role
    bit 0) and the decoded rows are candidates (role bit 1).  ``u`` [batch, r_max]
    float32 is drawn uniform in [0, 5) nats."""
    batch, seq_len = is_masked.shape
    role = np.zeros((batch, r_max), np.uint8)
    drafted = np.zeros((batch, seq_len), np.uint8)
    for b in range(batch):
        rows = np.arange(int(count[b]))
        masked = rows[is_masked[b, idx[b, rows]] != 0]
        pick = rng.choice(masked, size=min(n_drafted, len(masked)), replace=False)
        drafted[b, idx[b, pick]] = 1
        role[b, np.setdiff1d(masked, pick)] = 1
        role[b, rows[is_masked[b, idx[b, rows]] == 0]] = 2
    u = rng.uniform(0.0, 5.0, (batch, r_max)).astype(np.float32)
    return role, drafted, u


def scaled(w: Workload, **changes) -> Workload:
    """A copy of ``w`` with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **changes)


# ---------------------------------------------------------------------------
# element types


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _as_dtype(x32: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == BF16:
        return f32_to_bf16_bits(x32)
    if dtype == F32:
        return np.ascontiguousarray(x32, dtype=np.float32)
    raise ValueError(f"unsupported dtype code {dtype}")


# ---------------------------------------------------------------------------
# logits


def make_logits(rng: np.random.Generator, n_rows: int, vocab: int, dtype: int,
                near_uniform_frac: float = 0.0) -> np.ndarray:
    """``[n_rows, vocab]`` logits of the temperature + spike recipe above."""
    x = rng.standard_normal((n_rows, vocab), dtype=np.float32)
    n_near = int(round(near_uniform_frac * n_rows))
    order = rng.permutation(n_rows)
    near = np.zeros(n_rows, dtype=bool)
    near[order[:n_near]] = True
    t_spiked = np.exp(rng.uniform(math.log(0.1), math.log(3.0), size=n_rows)).astype(np.float32)
    t_near = np.exp(rng.uniform(math.log(5.0), math.log(20.0), size=n_rows)).astype(np.float32)
    spike = rng.uniform(0.0, 15.0, size=n_rows).astype(np.float32)
    spike_at = rng.integers(0, vocab, size=n_rows)
    for i in range(n_rows):
        if near[i]:
            x[i] /= t_near[i]
        else:
            x[i] *= t_spiked[i]
            x[i, spike_at[i]] += spike[i]
    return _as_dtype(x, dtype)


# ---------------------------------------------------------------------------
# decode state


@dataclasses.dataclass
class DecodeState:
    is_masked: np.ndarray    # uint8 [B, L]
    tokens: np.ndarray       # int32 [B, L]
    decode_step: np.ndarray  # int32 [B, L], -1 = never decoded
    step: int                # index of the denoising step about to run
    block_lo: int            # active block [block_lo, block_hi)
    block_hi: int
    row_pos: np.ndarray      # int32 [N]: position of each logits row
    seq_row_offsets: np.ndarray  # int32 [B + 1]


def make_state(rng: np.random.Generator, w: Workload) -> DecodeState:
    B, L, n = w.batch, w.seq_len, w.n_unmask
    gen0 = w.prompt_len
    lo = gen0 + w.active_block * w.block
    hi = lo + w.block
    if hi > L:
        raise ValueError("active block runs past the sequence")
    is_masked = np.zeros((B, L), np.uint8)
    tokens = rng.integers(0, w.vocab, size=(B, L)).astype(np.int32)
    decode_step = np.full((B, L), -1, np.int32)
    is_masked[:, lo:] = 1
    tokens[:, lo:] = w.vocab
    n_prev = lo - gen0
    for b in range(B):
        order = np.concatenate([gen0 + i * w.block + rng.permutation(w.block)
                                for i in range(w.active_block)]) if n_prev else np.zeros(0, int)
        decode_step[b, order] = (np.arange(n_prev) // n).astype(np.int32)
    step = (n_prev + n - 1) // n
    row_pos = np.concatenate([np.arange(lo, hi, dtype=np.int32) for _ in range(B)])
    offsets = (np.arange(B + 1, dtype=np.int32) * w.block).astype(np.int32)
    return DecodeState(is_masked, tokens, decode_step, step, lo, hi, row_pos, offsets)


# ---------------------------------------------------------------------------
# attention operands


@dataclasses.dataclass
class AttentionInputs:
    q: np.ndarray        # [B, r_max, H, d]
    k_new: np.ndarray    # [B, r_max, Hkv, d]
    v_new: np.ndarray
    k_cache: np.ndarray  # [B, L, Hkv, d] (pre-step)
    v_cache: np.ndarray
    dtype: int


def make_attention(rng: np.random.Generator, w: Workload, r_max: int,
                   std: float | None = None) -> AttentionInputs:
    s = w.qkv_std if std is None else std
    B, L, H, Hkv, d = w.batch, w.seq_len, w.n_heads, w.n_kv_heads, w.head_dim

    def draw(*shape):
        x = rng.standard_normal(shape, dtype=np.float32)
        x *= np.float32(s)
        return _as_dtype(x, w.attn_dtype)

    q = draw(B, r_max, H, d)
    k_new = draw(B, r_max, Hkv, d)
    v_new = draw(B, r_max, Hkv, d)
    k_cache = draw(B, L, Hkv, d)
    v_cache = draw(B, L, Hkv, d)
    return AttentionInputs(q, k_new, v_new, k_cache, v_cache, w.attn_dtype)


def make_lmhead(rng: np.random.Generator, n_rows: int, vocab: int, hidden: int,
                exact: bool = True) -> tuple[np.ndarray, np.ndarray]:
    """(hidden bf16 bits ``[n_rows, hidden]``, W_lm bf16 bits ``[vocab, hidden]``)
    of the LM-head recipes above."""
    w = np.empty((vocab, hidden), np.uint16)
    if exact:
        w_int = np.empty((vocab, hidden), np.int8)
        for r0 in range(0, vocab, 8192):
            r1 = min(vocab, r0 + 8192)
            w_int[r0:r1] = rng.integers(-3, 4, size=(r1 - r0, hidden), dtype=np.int8)
            w[r0:r1] = f32_to_bf16_bits(w_int[r0:r1].astype(np.float32) * np.float32(2.0 ** -6))
        m = max(1, hidden // 8)
        sigma = rng.choice(np.array([0.125, 0.25, 0.5, 1.0]), size=n_rows)
        spike = rng.choice(np.array([0.0, 2.0, 4.0, 8.0, 16.0]), size=n_rows,
                           p=[0.5, 0.15, 0.15, 0.15, 0.05])
        target = rng.integers(0, vocab, size=n_rows)
        x = np.empty((n_rows, hidden), np.uint16)
        for i in range(n_rows):
            a = int(round(6 + math.log2(sigma[i] / (4 * math.sqrt(hidden)))))
            row = rng.integers(-3, 4, size=hidden).astype(np.float64) * 2.0 ** a
            if spike[i] > 0:
                b = int(round(6 + math.log2(spike[i] / (4 * m))))
                b = min(max(b, a - 5), a + 5)
                on = rng.choice(hidden, size=m, replace=False)
                row[on] += w_int[target[i], on].astype(np.float64) * 2.0 ** b
            x[i] = f32_to_bf16_bits(row.astype(np.float32))
        return x, w
    std = np.float32(2.0 / math.sqrt(hidden))
    for r0 in range(0, vocab, 8192):
        r1 = min(vocab, r0 + 8192)
        w[r0:r1] = f32_to_bf16_bits(rng.standard_normal((r1 - r0, hidden), dtype=np.float32) * std)
    x = f32_to_bf16_bits(rng.standard_normal((n_rows, hidden), dtype=np.float32))
    return x, w


def random_index_set(rng: np.random.Generator, batch: int, seq_len: int,
                     counts: np.ndarray, stride: int) -> np.ndarray:
    """``[batch, stride]`` int32: row b holds ``counts[b]`` distinct positions in
    ascending order, the rest -1 (a generic recompute set for attention-only cases)."""
    idx = np.full((batch, stride), -1, np.int32)
    for b in range(batch):
        c = int(counts[b])
        idx[b, :c] = np.sort(rng.choice(seq_len, size=c, replace=False)).astype(np.int32)
    return idx


def step_rng(seed: int, step: int) -> np.random.Generator:
    """Independent generator for the logits of one trajectory step."""
    return np.random.default_rng(np.random.SeedSequence([seed, step]))


def random_state(rng: np.random.Generator, batch: int, seq_len: int, p_masked: float = 0.3,
                 max_step: int = 40):
    """Unstructured decode state for edge-case tests: each position masked with
    probability p_masked, otherwise prompt (-1) or decoded at a step in [0, max_step)."""
    is_masked = (rng.uniform(size=(batch, seq_len)) < p_masked).astype(np.uint8)
    steps = rng.integers(-1, max_step, size=(batch, seq_len)).astype(np.int32)
    decode_step = np.where(is_masked == 1, -1, steps).astype(np.int32)
    return is_masked, decode_step


# ---------------------------------------------------------------------------
# multi-step trajectory (synthetic layers)


def trajectory_rows_per_step(w: Workload) -> list[int]:
    """Masked rows of the active block at every step: each block starts fully
    masked and loses ``n_unmask`` positions per step."""
    per_block = -(-w.block // w.n_unmask)
    rows = []
    for t in range(w.n_steps):
        j = t % per_block
        rows.append(max(0, w.block - j * w.n_unmask))
    return rows


def trajectory_block(w: Workload, step: int) -> tuple[int, int]:
    """Active block [lo, hi) at a step (blocks are decoded left to right)."""
    per_block = -(-w.block // w.n_unmask)
    j = min(step // per_block, (w.seq_len - w.prompt_len) // w.block - 1)
    lo = w.prompt_len + j * w.block
    return lo, lo + w.block


@dataclasses.dataclass
class TrajectoryStart:
    is_masked: np.ndarray    # uint8 [1, L]: the generated region is masked
    tokens: np.ndarray       # int32 [1, L]: prompt tokens, then the [MASK] id (= vocab)
    decode_step: np.ndarray  # int32 [1, L]: -1 everywhere


def trajectory_start(seed: int, w: Workload) -> TrajectoryStart:
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x7A]))
    L = w.seq_len
    tokens = np.full((1, L), w.vocab, np.int32)
    tokens[0, :w.prompt_len] = rng.integers(0, w.vocab, size=w.prompt_len)
    is_masked = np.zeros((1, L), np.uint8)
    is_masked[0, w.prompt_len:] = 1
    return TrajectoryStart(is_masked, tokens, np.full((1, L), -1, np.int32))


def trajectory_layer_weights(seed: int, layer: int, hidden: int, ffn: int) -> dict:
    """bf16 weights of one pre-norm layer: w_qkv [3h, h], w_o [h, h], w_gu [2F, h]
    (gate rows, then up rows), w_down [h, F], each N(0, 1/fan_in); the two RMS-norm
    gains 1 + N(0, 0.1^2)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x1A7, layer]))

    def draw(rows, cols):
        x = rng.standard_normal((rows, cols), dtype=np.float32)
        x *= np.float32(1.0 / math.sqrt(cols))
        return f32_to_bf16_bits(x)

    gains = (1.0 + 0.1 * rng.standard_normal((2, hidden))).astype(np.float32)
    return dict(w_qkv=draw(3 * hidden, hidden), w_o=draw(hidden, hidden), w_gu=draw(2 * ffn, hidden),
                w_down=draw(hidden, ffn), g1=f32_to_bf16_bits(gains[0]), g2=f32_to_bf16_bits(gains[1]))


def trajectory_embedding(seed: int, vocab: int, hidden: int) -> np.ndarray:
    """bf16 ``[vocab + 1, hidden]`` N(0, 1) table; row ``vocab`` is the [MASK] input."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0xE3]))
    return f32_to_bf16_bits(rng.standard_normal((vocab + 1, hidden), dtype=np.float32))


def trajectory_weights(seed: int, layer: int, hidden: int, width: int) -> np.ndarray:
    """bf16 ``[3 width, hidden]`` N(0, 1/hidden) weights [W_q; W_k; W_v] of one layer."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x3E, layer]))
    x = rng.standard_normal((3 * width, hidden), dtype=np.float32)
    x *= np.float32(1.0 / math.sqrt(hidden))
    return f32_to_bf16_bits(x)


def trajectory_logits(seed: int, step: int, n_rows: int, vocab: int) -> np.ndarray:
    """bf16 logits of one step's masked rows (the temperature + spike recipe)."""
    return make_logits(step_rng(seed, step), n_rows, vocab, BF16)


def trajectory_window_logits(seed: int, step: int, width: int, vocab: int) -> np.ndarray:
    """bf16 logits of ``width`` rows for one step of a window-policy trajectory; a
    step whose window holds c masked positions uses the first c rows."""
    return make_logits(step_rng(seed, step), width, vocab, BF16)
