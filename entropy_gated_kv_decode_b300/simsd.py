"""SimSD's input layout on the host: the rotary positions of its rows.

"SimSD - Simple Speculative Decoding in Diffusion Language Models", Italian
technical summary, "Metodologia: SimSD", item 3 (RoPE copy): every prediction
slot of the mask section reuses the rotary index of the data token of the same
response position, so the model sees the reference token and its slot at one
position.  With the layout of item 1 (prompt of P positions, data section, mask
section, B positions each) slot P + B + k takes rotary position P + k; every
other position keeps its own.  The result is the per-row position array that
ec_rope takes in place of the rows' sequence positions.
"""
from __future__ import annotations

import numpy as np


def rope_positions(idx: np.ndarray, count: np.ndarray, prompt_len: int, block: int) -> np.ndarray:
    """int32 [B, stride]: the rotary position of every row (rows past count keep
    their entries)."""
    pos = np.array(idx, dtype=np.int32, copy=True)
    slots = (pos >= prompt_len + block) & (pos < prompt_len + 2 * block)
    live = np.arange(pos.shape[1])[None, :] < np.asarray(count)[:, None]
    pos[slots & live] -= block
    return pos
