"""Shared plumbing for the GPU parity tests: upload the generator's host arrays,
run the CUDA path through the binding, run the oracle on the same arrays, and
compare with the tolerances the method's decisions allow."""
from __future__ import annotations

import math

import numpy as np
import torch

from entropy_gated_kv_decode_b300 import synth

ENTROPY_ATOL = 1e-4      # nats
CONF_RTOL = 2e-5
GATE_MARGIN = 1e-4       # |E - tau| below this: decision excluded and reported
TIE_RTOL = 1e-6          # confidences closer than this are a near tie
ATTN_RTOL, ATTN_ATOL = 2e-2, 1e-2   # bf16
ATTN_F32_TOL = 1e-4


def native():
    from entropy_gated_kv_decode_b300 import build, _native
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return _native


def dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def run_decode_gpu(nat, logits: np.ndarray, state: synth.DecodeState, n_unmask: int, tau: float,
                   step: int, row_stride: int | None = None, workspace=None):
    """One ec_decode_step on a copy of the state; returns host arrays."""
    n_rows, vocab = logits.shape
    B, L = state.is_masked.shape
    if row_stride is not None and row_stride != vocab:
        padded = np.zeros((n_rows, row_stride), logits.dtype)
        padded[:, :vocab] = logits
        lg = dev(padded)[:, :vocab]
    else:
        lg = dev(logits)
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
        nat.ec_decode_workspace_size(n_rows, B))
    nat.ec_decode_step(lg, dev(state.seq_row_offsets), dev(state.row_pos), L, n_unmask, tau, step,
                       out["token"], out["conf"], out["entropy"], out["unmask_rows"],
                       out["max_entropy"], out["refresh"], im, tk, ds, ws)
    bits = nat.ec_read_device_status(ws)
    res = {k: host(v) for k, v in out.items()}
    res["unmask_rows"] = res["unmask_rows"].reshape(B, n_unmask)
    res.update(is_masked=host(im), tokens=host(tk), decode_step=host(ds), status=bits)
    return res


def run_decode_oracle(orc, logits, state, n_unmask, tau, step):
    h, c, t = orc.row_stats(logits)
    g = orc.unmask_gate(c, h, t, state.seq_row_offsets, state.row_pos, state.is_masked.shape[1],
                        n_unmask, tau, step, state.is_masked, state.tokens, state.decode_step)
    g.update(entropy=h, conf=c, token=t)
    return g


def check_decode(gpu, ref, state, n_unmask, tau, step):
    """Compare; returns the set of sequences whose decisions were excluded
    (near tie in the unmask order or |E - tau| < GATE_MARGIN)."""
    tau32 = float(np.float32(tau))
    assert gpu["status"] == 0, f"device status bits {gpu['status']:#x}"
    # per row
    assert np.array_equal(gpu["token"], ref["token"]), "argmax tokens differ"
    assert np.all(np.abs(gpu["entropy"] - ref["entropy"]) <= ENTROPY_ATOL), \
        f"entropy error {np.max(np.abs(gpu['entropy'] - ref['entropy']))}"
    assert np.allclose(gpu["conf"], ref["conf"], rtol=CONF_RTOL, atol=0)
    excluded = set()
    off = state.seq_row_offsets
    B = len(off) - 1
    for b in range(B):
        rows = np.arange(off[b], off[b + 1])
        g_sel = [r for r in gpu["unmask_rows"][b] if r >= 0]
        o_sel = [r for r in ref["unmask_rows"][b] if r >= 0]
        # the GPU order is exactly its own confidences ranked (ties: lower position)
        own = sorted(rows.tolist(), key=lambda r: (-gpu["conf"][r], state.row_pos[r]))[:n_unmask]
        assert g_sel == own, f"seq {b}: GPU unmask order is not its own ranking"
        assert list(gpu["unmask_rows"][b][len(g_sel):]) == [-1] * (n_unmask - len(g_sel))
        # internal gate consistency
        e_gpu = max((gpu["entropy"][r] for r in g_sel), default=-math.inf)
        assert gpu["max_entropy"][b] == np.float32(e_gpu)
        assert gpu["refresh"][b] == (1 if gpu["max_entropy"][b] > np.float32(tau) else 0)
        if g_sel != o_sel:
            c = ref["conf"]
            lo = min(c[r] for r in g_sel) if g_sel else math.inf
            others = [r for r in rows if r not in g_sel]
            valid = all(c[g_sel[i]] >= c[g_sel[i + 1]] * (1 - TIE_RTOL) for i in range(len(g_sel) - 1))
            valid &= all(c[u] <= lo * (1 + TIE_RTOL) for u in others)
            assert valid, f"seq {b}: unmask order {g_sel} vs oracle {o_sel} is not a near tie"
            excluded.add(b)
            continue
        if abs(ref["max_entropy"][b] - tau32) < GATE_MARGIN:
            excluded.add(b)
        else:
            assert gpu["refresh"][b] == ref["refresh"][b], f"seq {b}: refresh differs"
        if np.isfinite(ref["max_entropy"][b]):
            assert abs(gpu["max_entropy"][b] - ref["max_entropy"][b]) <= ENTROPY_ATOL
        else:
            assert gpu["max_entropy"][b] == -np.inf
        for name in ("is_masked", "tokens", "decode_step"):
            assert np.array_equal(gpu[name][b], ref[name][b]), f"seq {b}: {name} differs"
    return excluded


def run_recompute_gpu(nat, is_masked, decode_step, refresh, lo, hi, k):
    B, L = is_masked.shape
    idx = torch.full((B, L), -9, dtype=torch.int32, device="cuda")
    cnt = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    nat.ec_build_recompute_set(dev(is_masked), dev(decode_step), dev(refresh), lo, hi, k, idx, cnt)
    torch.cuda.synchronize()
    return host(idx), host(cnt)


def attention_close(gpu: np.ndarray, ref: np.ndarray, bf16: bool):
    """Elementwise rtol/atol and a per-(row, head) relative Frobenius bound."""
    if gpu.size == 0:
        return
    if bf16:
        ok = np.abs(gpu - ref) <= ATTN_ATOL + ATTN_RTOL * np.abs(ref)
        assert ok.all(), f"attention max abs error {np.max(np.abs(gpu - ref))}"
        num = np.linalg.norm((gpu - ref).reshape(-1, ref.shape[-1]), axis=1)
        den = np.linalg.norm(ref.reshape(-1, ref.shape[-1]), axis=1) + 1e-30
        assert np.max(num / den) <= ATTN_RTOL, f"relative error {np.max(num / den)}"
    else:
        assert np.allclose(gpu, ref, rtol=ATTN_F32_TOL, atol=ATTN_F32_TOL), \
            f"attention max abs error {np.max(np.abs(gpu - ref))}"


def widen(a: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)
