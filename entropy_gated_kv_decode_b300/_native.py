"""Thin ctypes binding of ``libec.so`` (declared in ``include/ec.h``).

Argument marshalling only: every function checks that the tensors it is given
are CUDA tensors of the expected dtype and layout, passes their device
pointers, sizes and the current CUDA stream to the C function of the same
name, and raises ``ECError`` on a non-zero status.  All arithmetic runs in the
library's kernels; there is no other code path.  If the library has not been
built, every call raises ``NativeLibraryMissing``.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIBRARY = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libec.so")

EC_F32, EC_BF16 = 0, 1
WORKSPACE_ALIGN = 256

DEV_BAD_OFFSETS = 0x1
DEV_BAD_ROW_POS = 0x2
DEV_BAD_COUNT = 0x4
DEV_BAD_INDEX = 0x8
DEV_TIMEOUT = 0x10
DEV_BAD_LABEL = 0x20

EXPORTED = ("ec_status_str", "ec_abi_version", "ec_debug_set_wait_limit", "ec_workspace_init",
            "ec_read_device_status",
            "ec_decode_workspace_size", "ec_decode_step", "ec_decode_step_noalloc",
            "ec_decode_noalloc_read_status", "ec_lmhead_workspace_size", "ec_lmhead_decode_step",
            "ec_build_recompute_set", "ec_attention_workspace_size", "ec_attention_kernel_count",
            "ec_selective_attention", "ec_selective_attention_simsd",
            "ec_selective_attention_cover", "ec_embed_rows", "ec_qkv_projection",
            "ec_rms_norm", "ec_rope", "ec_linear",
            "ec_cover_score_workspace_size", "ec_cover_seed_score", "ec_cover_score_kernel_count")


class NativeLibraryMissing(RuntimeError):
    pass


class ECError(RuntimeError):
    def __init__(self, code: int, fn: str):
        self.code = code
        super().__init__(f"{fn}: {status_str(code)} ({code})")


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            raise NativeLibraryMissing(
                f"{LIBRARY} is missing; build it with `python -m entropy_gated_kv_decode_b300.build`")
        L = ctypes.CDLL(LIBRARY)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t)
        L.ec_status_str.argtypes = [ctypes.c_int]
        L.ec_status_str.restype = ctypes.c_char_p
        L.ec_abi_version.argtypes = []
        L.ec_abi_version.restype = ctypes.c_int
        L.ec_debug_set_wait_limit.argtypes = [i64]
        L.ec_workspace_init.argtypes = [vp, sz, vp]
        L.ec_read_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
        L.ec_decode_workspace_size.argtypes = [i32, i32]
        L.ec_decode_workspace_size.restype = sz
        L.ec_decode_step.argtypes = [vp, ctypes.c_int, i64, i32, i32, vp, vp, i32, i32, i32, f32,
                                     i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ec_decode_step_noalloc.argtypes = [vp, ctypes.c_int, i64, i32, i32, vp, vp, i32, i32, i32,
                                             f32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.ec_decode_noalloc_read_status.argtypes = [vp, vp]
        L.ec_lmhead_workspace_size.argtypes = [i32, i32, i32]
        L.ec_lmhead_workspace_size.restype = sz
        L.ec_lmhead_decode_step.argtypes = [vp, vp, i32, i32, i32, vp, vp, i32, i32, i32, f32, i32,
                                            vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ec_build_recompute_set.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
        L.ec_attention_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        L.ec_attention_workspace_size.restype = sz
        L.ec_attention_kernel_count.argtypes = [ctypes.c_int, i32, i32, i32, i32, i32, i32]
        L.ec_attention_kernel_count.restype = i32
        L.ec_selective_attention.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, vp, ctypes.c_int,
                                             i32, i32, i32, i32, i32, i32, f32, vp, sz, vp]
        L.ec_selective_attention_simsd.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp,
                                                   ctypes.c_int, i32, i32, i32, i32, i32, i32, f32,
                                                   vp, sz, vp]
        L.ec_selective_attention_cover.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, vp, vp,
                                                   ctypes.c_int, i32, i32, i32, i32, i32, i32, f32,
                                                   vp, sz, vp]
        L.ec_embed_rows.argtypes = [vp, i64, i32, vp, i64, vp, vp, vp, i32, i32, i32, i32, vp, vp,
                                    sz, vp]
        L.ec_qkv_projection.argtypes = [vp, vp, i32, i32, i32, vp, i32, vp, vp, vp, vp, sz, vp]
        L.ec_rms_norm.argtypes = [vp, vp, i32, i32, i32, vp, f32, vp, vp, sz, vp]
        L.ec_rope.argtypes = [vp, vp, vp, i64, vp, i32, i32, i32, i32, i32, i32, ctypes.c_double,
                              vp, sz, vp]
        L.ec_linear.argtypes = [vp, vp, i32, i32, i32, vp, i32, i32, vp, vp, vp, sz, vp]
        L.ec_cover_score_workspace_size.argtypes = [i32, i32, i32, i32]
        L.ec_cover_score_workspace_size.restype = sz
        L.ec_cover_seed_score.argtypes = [vp, vp, vp, i64, vp, vp, vp, vp, ctypes.c_int, i32, i32,
                                          i32, i32, i32, i32, f32, i32, vp, vp, vp, vp, vp, sz, vp]
        L.ec_cover_score_kernel_count.argtypes = [i32, i32, i32]
        L.ec_cover_score_kernel_count.restype = i32
        for name in ("ec_debug_set_wait_limit", "ec_workspace_init", "ec_read_device_status",
                     "ec_decode_step",
                     "ec_decode_step_noalloc", "ec_decode_noalloc_read_status",
                     "ec_lmhead_decode_step", "ec_build_recompute_set",
                     "ec_selective_attention", "ec_selective_attention_simsd",
                     "ec_selective_attention_cover", "ec_embed_rows", "ec_qkv_projection",
                     "ec_rms_norm", "ec_rope", "ec_linear", "ec_cover_seed_score"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def status_str(code: int) -> str:
    return lib().ec_status_str(code).decode()


def _check(rc: int, fn: str):
    if rc != 0:
        raise ECError(rc, fn)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(name, t, dtype=None, contiguous=True):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _float_code(t):
    if t.dtype == torch.bfloat16:
        return EC_BF16
    if t.dtype == torch.float32:
        return EC_F32
    raise TypeError(f"unsupported dtype {t.dtype}: float32 or bfloat16")


def _numel(t, n, name):
    if t.numel() != n:
        raise ValueError(f"{name} must hold {n} elements, has {t.numel()}")


# ---------------------------------------------------------------------------


def ec_abi_version() -> int:
    return lib().ec_abi_version()


def ec_decode_workspace_size(n_rows: int, batch: int) -> int:
    return lib().ec_decode_workspace_size(n_rows, batch)


def ec_attention_workspace_size(batch, seq_len, r_max, n_heads, n_kv_heads, head_dim) -> int:
    return lib().ec_attention_workspace_size(batch, seq_len, r_max, n_heads, n_kv_heads, head_dim)


def ec_attention_kernel_count(dtype, batch, seq_len, r_max, n_heads, n_kv_heads, head_dim) -> int:
    """Kernels one ec_selective_attention call launches (dtype: torch.bfloat16 or
    torch.float32); -1 for arguments the call rejects."""
    code = {torch.bfloat16: EC_BF16, torch.float32: EC_F32}[dtype]
    return lib().ec_attention_kernel_count(code, batch, seq_len, r_max, n_heads, n_kv_heads,
                                           head_dim)


def ec_debug_set_wait_limit(cycles: int):
    """Test hook: the cycle limit of every in-kernel wait of later launches
    (0 restores the default of about 2 s); see ec.h."""
    _check(lib().ec_debug_set_wait_limit(int(cycles)), "ec_debug_set_wait_limit")


def new_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zeroed device workspace (torch's allocator returns 512-byte aligned blocks)."""
    ws = torch.zeros(max(int(nbytes), WORKSPACE_ALIGN), dtype=torch.uint8, device=device)
    if ws.data_ptr() % WORKSPACE_ALIGN:
        raise RuntimeError("workspace allocation is not 256-byte aligned")
    return ws


def ec_workspace_init(workspace: torch.Tensor, stream=None):
    _cuda("workspace", workspace, torch.uint8)
    _check(lib().ec_workspace_init(_p(workspace), workspace.numel(), _stream(stream)),
           "ec_workspace_init")


def ec_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    _cuda("workspace", workspace, torch.uint8)
    bits = ctypes.c_uint32(0)
    _check(lib().ec_read_device_status(_p(workspace), ctypes.byref(bits), _stream(stream)),
           "ec_read_device_status")
    return bits.value


def _decode_args(logits, seq_row_offsets, row_pos, seq_len, n_unmask, tau, step, token_out,
                 conf_out, entropy_out, unmask_rows, max_entropy, refresh, is_masked, seq_tokens,
                 decode_step, workspace=None):
    """Arguments of ec_decode_step (workspace given) or of ec_decode_step_noalloc
    (workspace None: no workspace arguments)."""
    _cuda("logits", logits, contiguous=False)
    if logits.dim() != 2 or (logits.shape[0] > 0 and logits.stride(1) != 1):
        raise ValueError("logits must be [N, V] with unit stride along V")
    n_rows, vocab = logits.shape
    batch = seq_row_offsets.numel() - 1
    _cuda("seq_row_offsets", seq_row_offsets, torch.int32)
    _cuda("row_pos", row_pos, torch.int32)
    for name, t, dt, n in (("token_out", token_out, torch.int32, n_rows),
                           ("conf_out", conf_out, torch.float32, n_rows),
                           ("entropy_out", entropy_out, torch.float32, n_rows),
                           ("unmask_rows", unmask_rows, torch.int32, batch * n_unmask),
                           ("max_entropy", max_entropy, torch.float32, batch),
                           ("refresh", refresh, torch.uint8, batch),
                           ("is_masked", is_masked, torch.uint8, batch * seq_len),
                           ("seq_tokens", seq_tokens, torch.int32, batch * seq_len),
                           ("decode_step", decode_step, torch.int32, batch * seq_len)):
        _cuda(name, t, dt)
        _numel(t, n, name)
    _numel(row_pos, n_rows, "row_pos")
    args = [_p(logits), _float_code(logits), logits.stride(0) if n_rows > 0 else vocab, n_rows,
            vocab, _p(seq_row_offsets), _p(row_pos), batch, seq_len, n_unmask, float(tau),
            int(step), _p(token_out), _p(conf_out), _p(entropy_out), _p(unmask_rows),
            _p(max_entropy), _p(refresh), _p(is_masked), _p(seq_tokens), _p(decode_step)]
    if workspace is not None:
        _cuda("workspace", workspace, torch.uint8)
        args += [_p(workspace), workspace.numel()]
    return args


def ec_decode_step(logits, seq_row_offsets, row_pos, seq_len, n_unmask, tau, step,
                   token_out, conf_out, entropy_out, unmask_rows, max_entropy, refresh,
                   is_masked, seq_tokens, decode_step, workspace, stream=None):
    """logits [N, V] (row stride may exceed V); see ``ec_decode_step`` in ec.h."""
    args = _decode_args(logits, seq_row_offsets, row_pos, seq_len, n_unmask, tau, step,
                        token_out, conf_out, entropy_out, unmask_rows, max_entropy, refresh,
                        is_masked, seq_tokens, decode_step, workspace)
    _check(lib().ec_decode_step(*args, _stream(stream)), "ec_decode_step")


def ec_decode_step_noalloc(logits, seq_row_offsets, row_pos, seq_len, n_unmask, tau, step,
                           token_out, conf_out, entropy_out, unmask_rows, max_entropy, refresh,
                           is_masked, seq_tokens, decode_step, stream=None):
    """ec_decode_step without a workspace, for callers that cannot allocate device
    memory: the scratch is a fixed 2 MiB array inside the library (see ec.h)."""
    args = _decode_args(logits, seq_row_offsets, row_pos, seq_len, n_unmask, tau, step,
                        token_out, conf_out, entropy_out, unmask_rows, max_entropy, refresh,
                        is_masked, seq_tokens, decode_step)
    _check(lib().ec_decode_step_noalloc(*args, _stream(stream)), "ec_decode_step_noalloc")


def ec_decode_noalloc_read_status(stream=None) -> int:
    """Device status bits of the last ec_decode_step_noalloc call on this device."""
    bits = ctypes.c_uint32(0)
    _check(lib().ec_decode_noalloc_read_status(ctypes.byref(bits), _stream(stream)),
           "ec_decode_noalloc_read_status")
    return bits.value


def ec_lmhead_workspace_size(n_rows: int, vocab: int, batch: int) -> int:
    return lib().ec_lmhead_workspace_size(n_rows, vocab, batch)


def _lmhead_args(hidden, w_lm, seq_row_offsets, row_pos, seq_len, n_unmask, tau, step, token_out,
                 conf_out, entropy_out, unmask_rows, max_entropy, refresh, is_masked, seq_tokens,
                 decode_step, workspace):
    _cuda("hidden", hidden, torch.bfloat16)
    _cuda("w_lm", w_lm, torch.bfloat16)
    if hidden.dim() != 2 or w_lm.dim() != 2 or hidden.shape[1] != w_lm.shape[1]:
        raise ValueError("hidden must be [N, hidden_dim] and w_lm [vocab, hidden_dim]")
    n_rows, hidden_dim = hidden.shape
    vocab = w_lm.shape[0]
    batch = seq_row_offsets.numel() - 1
    _cuda("seq_row_offsets", seq_row_offsets, torch.int32)
    _cuda("row_pos", row_pos, torch.int32)
    for name, t, dt, n in (("token_out", token_out, torch.int32, n_rows),
                           ("conf_out", conf_out, torch.float32, n_rows),
                           ("entropy_out", entropy_out, torch.float32, n_rows),
                           ("unmask_rows", unmask_rows, torch.int32, batch * n_unmask),
                           ("max_entropy", max_entropy, torch.float32, batch),
                           ("refresh", refresh, torch.uint8, batch),
                           ("is_masked", is_masked, torch.uint8, batch * seq_len),
                           ("seq_tokens", seq_tokens, torch.int32, batch * seq_len),
                           ("decode_step", decode_step, torch.int32, batch * seq_len)):
        _cuda(name, t, dt)
        _numel(t, n, name)
    _numel(row_pos, n_rows, "row_pos")
    _cuda("workspace", workspace, torch.uint8)
    return [_p(hidden), _p(w_lm), n_rows, hidden_dim, vocab, _p(seq_row_offsets), _p(row_pos),
            batch, seq_len, n_unmask, float(tau), int(step), _p(token_out), _p(conf_out),
            _p(entropy_out), _p(unmask_rows), _p(max_entropy), _p(refresh), _p(is_masked),
            _p(seq_tokens), _p(decode_step), _p(workspace), workspace.numel()]


def ec_lmhead_decode_step(hidden, w_lm, seq_row_offsets, row_pos, seq_len, n_unmask, tau, step,
                          token_out, conf_out, entropy_out, unmask_rows, max_entropy, refresh,
                          is_masked, seq_tokens, decode_step, workspace, stream=None):
    """hidden [N, hidden_dim] and w_lm [vocab, hidden_dim] bf16; the decode-and-gate
    step on the logits hidden @ w_lm.T, which are never materialised (see ec.h)."""
    args = _lmhead_args(hidden, w_lm, seq_row_offsets, row_pos, seq_len, n_unmask, tau, step,
                        token_out, conf_out, entropy_out, unmask_rows, max_entropy, refresh,
                        is_masked, seq_tokens, decode_step, workspace)
    _check(lib().ec_lmhead_decode_step(*args, _stream(stream)), "ec_lmhead_decode_step")


def _recompute_args(is_masked, decode_step, refresh, block_lo, block_hi, k, idx, count):
    _cuda("is_masked", is_masked, torch.uint8)
    _cuda("decode_step", decode_step, torch.int32)
    _cuda("refresh", refresh, torch.uint8)
    _cuda("idx", idx, torch.int32)
    _cuda("count", count, torch.int32)
    batch, seq_len = is_masked.shape
    for name, t, n in (("decode_step", decode_step, batch * seq_len), ("refresh", refresh, batch),
                       ("idx", idx, batch * seq_len), ("count", count, batch)):
        _numel(t, n, name)
    return [_p(is_masked), _p(decode_step), _p(refresh), batch, seq_len, block_lo, block_hi, k,
            _p(idx), _p(count)]


def ec_build_recompute_set(is_masked, decode_step, refresh, block_lo, block_hi, k, idx, count,
                           stream=None):
    """is_masked / decode_step [B, L]; idx [B, L] and count [B] are written."""
    args = _recompute_args(is_masked, decode_step, refresh, block_lo, block_hi, k, idx, count)
    _check(lib().ec_build_recompute_set(*args, _stream(stream)), "ec_build_recompute_set")


def _attention_args(q, k_new, v_new, idx, count, k_cache, v_cache, out, scale, workspace):
    for name, t in (("q", q), ("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache),
                    ("v_cache", v_cache), ("out", out)):
        _cuda(name, t, q.dtype)
    _cuda("idx", idx, torch.int32)
    _cuda("count", count, torch.int32)
    _cuda("workspace", workspace, torch.uint8)
    batch, r_max, n_heads, head_dim = q.shape
    seq_len, n_kv = k_cache.shape[1], k_cache.shape[2]
    if (k_new.shape != (batch, r_max, n_kv, head_dim) or v_new.shape != k_new.shape
            or k_cache.shape != (batch, seq_len, n_kv, head_dim) or v_cache.shape != k_cache.shape
            or out.shape != q.shape or idx.dim() != 2 or idx.shape[0] != batch
            or count.numel() != batch):
        raise ValueError("inconsistent attention shapes")
    return [_p(q), _p(k_new), _p(v_new), _p(idx), idx.shape[1], _p(count), _p(k_cache),
            _p(v_cache), _p(out), _float_code(q), batch, seq_len, r_max, n_heads, n_kv, head_dim,
            float(scale), _p(workspace), workspace.numel()]


def ec_selective_attention(q, k_new, v_new, idx, count, k_cache, v_cache, out, scale, workspace,
                           stream=None):
    """q/out [B, R, H, d]; k_new/v_new [B, R, Hkv, d]; caches [B, L, Hkv, d];
    idx [B, >= R] int32 (row stride = its second dimension); count [B]."""
    args = _attention_args(q, k_new, v_new, idx, count, k_cache, v_cache, out, scale, workspace)
    _check(lib().ec_selective_attention(*args, _stream(stream)), "ec_selective_attention")


def _simsd_args(q, k_new, v_new, idx, count, section, tau, k_cache, v_cache, out, scale,
                workspace):
    a = _attention_args(q, k_new, v_new, idx, count, k_cache, v_cache, out, scale, workspace)
    _cuda("section", section, torch.uint8)
    _cuda("tau", tau, torch.int32)
    if section.shape != k_cache.shape[:2] or tau.shape != k_cache.shape[:2]:
        raise ValueError("section and tau must be [batch, seq_len]")
    return a[:6] + [_p(section), _p(tau)] + a[6:]


def ec_selective_attention_simsd(q, k_new, v_new, idx, count, section, tau, k_cache, v_cache,
                                 out, scale, workspace, stream=None):
    """ec_selective_attention under SimSD's temporal causal mask: section uint8 and
    tau int32 [B, L] (0 prompt, 1 data, 2 mask slot; step labels >= 1)."""
    args = _simsd_args(q, k_new, v_new, idx, count, section, tau, k_cache, v_cache, out, scale,
                       workspace)
    _check(lib().ec_selective_attention_simsd(*args, _stream(stream)),
           "ec_selective_attention_simsd")


def _cover_args(q, k_new, v_new, idx, count, seed, k_cache, v_cache, out, scale, workspace):
    a = _attention_args(q, k_new, v_new, idx, count, k_cache, v_cache, out, scale, workspace)
    _cuda("seed", seed, torch.uint8)
    if seed.shape != q.shape[:2]:
        raise ValueError("seed must be [batch, r_max]")
    return a[:6] + [_p(seed)] + a[6:]


def ec_selective_attention_cover(q, k_new, v_new, idx, count, seed, k_cache, v_cache, out,
                                 scale, workspace, stream=None):
    """ec_selective_attention with COVER's dual view: seed uint8 [B, R] flags the
    recomputed rows that are seeds (masked-input K/V, not written back)."""
    args = _cover_args(q, k_new, v_new, idx, count, seed, k_cache, v_cache, out, scale, workspace)
    _check(lib().ec_selective_attention_cover(*args, _stream(stream)),
           "ec_selective_attention_cover")


def ec_cover_score_workspace_size(batch, seq_len, r_max, n_heads) -> int:
    return int(lib().ec_cover_score_workspace_size(batch, seq_len, r_max, n_heads))


def ec_cover_score_kernel_count(batch, r_max, n_seed) -> int:
    return int(lib().ec_cover_score_kernel_count(batch, r_max, n_seed))


def _cover_score_args(q, k_cache, idx, count, role, drafted, u, scale, n_seed, d_in, d_out, score,
                      seeds, workspace):
    _cuda("q", q, torch.bfloat16)
    _cuda("k_cache", k_cache, torch.bfloat16)
    _cuda("idx", idx, torch.int32)
    _cuda("count", count, torch.int32)
    _cuda("role", role, torch.uint8)
    _cuda("drafted", drafted, torch.uint8)
    for name, t in (("u", u), ("d_in", d_in), ("d_out", d_out), ("score", score)):
        _cuda(name, t, torch.float32)
    _cuda("workspace", workspace, torch.uint8)
    if q.dim() != 4 or k_cache.dim() != 4:
        raise ValueError("q must be [B, R, H, d] and k_cache [B, L, Hkv, d]")
    batch, r_max, n_heads, head_dim = q.shape
    seq_len, n_kv_heads = k_cache.shape[1], k_cache.shape[2]
    n_seed = int(n_seed)
    if (k_cache.shape[0] != batch or k_cache.shape[3] != head_dim or idx.dim() != 2
            or idx.shape[0] != batch or count.numel() != batch
            or tuple(role.shape) != (batch, r_max) or tuple(u.shape) != (batch, r_max)
            or tuple(drafted.shape) != (batch, seq_len)
            or any(tuple(t.shape) != (batch, r_max) for t in (d_in, d_out, score))):
        raise ValueError("inconsistent seed-score shapes")
    if n_seed > 0:
        _cuda("seeds", seeds, torch.int32)
        if tuple(seeds.shape) != (batch, n_seed):
            raise ValueError("seeds must be [B, n_seed]")
    return [_p(q), _p(k_cache), _p(idx), idx.shape[1], _p(count), _p(role), _p(drafted), _p(u),
            EC_BF16, batch, seq_len, r_max, n_heads, n_kv_heads, head_dim, float(scale), n_seed,
            _p(d_in), _p(d_out), _p(score), _p(seeds) if n_seed > 0 else None, _p(workspace),
            workspace.numel()]


def ec_cover_seed_score(q, k_cache, idx, count, role, drafted, u, scale, n_seed, d_in, d_out, score,
                        seeds, workspace, stream=None):
    """COVER's seed score: d_in, d_out, score [B, R] float32 at the candidate rows
    (role bit 1; bit 0 marks still-masked queries), seeds [B, n_seed] int32 positions."""
    args = _cover_score_args(q, k_cache, idx, count, role, drafted, u, scale, n_seed, d_in, d_out,
                             score, seeds, workspace)
    _check(lib().ec_cover_seed_score(*args, _stream(stream)), "ec_cover_seed_score")


def _embed_args(table, idx, count, seq_tokens, is_masked, mask_id, x, workspace):
    _cuda("table", table, torch.bfloat16)
    _cuda("idx", idx, torch.int32)
    _cuda("count", count, torch.int32)
    _cuda("seq_tokens", seq_tokens, torch.int32)
    _cuda("is_masked", is_masked, torch.uint8)
    _cuda("x", x, torch.bfloat16)
    _cuda("workspace", workspace, torch.uint8)
    batch, seq_len = seq_tokens.shape
    r_max, hidden = x.shape[-2], x.shape[-1]
    if (table.dim() != 2 or table.shape[1] != hidden or x.numel() != batch * r_max * hidden
            or idx.dim() != 2 or idx.shape[0] != batch or count.numel() != batch
            or is_masked.shape != seq_tokens.shape):
        raise ValueError("inconsistent embedding shapes")
    return [_p(table), table.shape[0], hidden, _p(idx), idx.shape[1], _p(count), _p(seq_tokens),
            _p(is_masked), int(mask_id), batch, seq_len, r_max, _p(x), _p(workspace),
            workspace.numel()]


def ec_embed_rows(table, idx, count, seq_tokens, is_masked, mask_id, x, workspace, stream=None):
    """x [B, r_max, hidden] <- table rows of the tokens at idx (mask_id while masked)."""
    args = _embed_args(table, idx, count, seq_tokens, is_masked, mask_id, x, workspace)
    _check(lib().ec_embed_rows(*args, _stream(stream)), "ec_embed_rows")


def _projection_args(x, count, w_qkv, q, k, v, workspace):
    for name, t in (("x", x), ("w_qkv", w_qkv), ("q", q), ("k", k), ("v", v)):
        _cuda(name, t, torch.bfloat16)
    _cuda("workspace", workspace, torch.uint8)
    if count is not None:
        _cuda("count", count, torch.int32)
    if x.dim() != 3:
        raise ValueError("x must be [batch, r_max, hidden]")
    batch, r_max, hidden = x.shape
    if w_qkv.dim() != 2 or w_qkv.shape[1] != hidden or w_qkv.shape[0] % 3:
        raise ValueError("w_qkv must be [3 * width, hidden]")
    width = w_qkv.shape[0] // 3
    for name, t in (("q", q), ("k", k), ("v", v)):
        _numel(t, batch * r_max * width, name)
    if count is not None:
        _numel(count, batch, "count")
    return [_p(x), _p(count), batch, r_max, hidden, _p(w_qkv), width, _p(q), _p(k), _p(v),
            _p(workspace), workspace.numel()]


def ec_qkv_projection(x, count, w_qkv, q, k, v, workspace, stream=None):
    """q/k/v [B, r_max, width] <- x [B, r_max, hidden] @ w_qkv[3 width, hidden]^T, rows < count."""
    args = _projection_args(x, count, w_qkv, q, k, v, workspace)
    _check(lib().ec_qkv_projection(*args, _stream(stream)), "ec_qkv_projection")


def _rms_norm_args(x, count, weight, eps, y, workspace):
    for name, t in (("x", x), ("weight", weight), ("y", y)):
        _cuda(name, t, torch.bfloat16)
    _cuda("workspace", workspace, torch.uint8)
    if count is not None:
        _cuda("count", count, torch.int32)
    if x.dim() != 3 or y.shape != x.shape or weight.numel() != x.shape[2]:
        raise ValueError("x, y [batch, r_max, hidden]; weight [hidden]")
    batch, r_max, hidden = x.shape
    return [_p(x), _p(count), batch, r_max, hidden, _p(weight), float(eps), _p(y), _p(workspace),
            workspace.numel()]


def ec_rms_norm(x, count, weight, eps, y, workspace, stream=None):
    """y = x / sqrt(mean(x^2) + eps) * weight over the rows < count (bf16)."""
    _check(lib().ec_rms_norm(*_rms_norm_args(x, count, weight, eps, y, workspace),
                             _stream(stream)), "ec_rms_norm")


def _rope_args(q, k, idx, count, seq_len, theta, workspace):
    for name, t in (("q", q), ("k", k)):
        _cuda(name, t, torch.bfloat16)
    _cuda("idx", idx, torch.int32)
    _cuda("count", count, torch.int32)
    _cuda("workspace", workspace, torch.uint8)
    if q.dim() != 4 or k.dim() != 4 or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q [batch, r_max, heads, d], k [batch, r_max, kv_heads, d]")
    batch, r_max, h, d = q.shape
    return [_p(q), _p(k), _p(idx), idx.shape[1], _p(count), batch, int(seq_len), r_max, h,
            k.shape[2], d, float(theta), _p(workspace), workspace.numel()]


def ec_rope(q, k, idx, count, seq_len, theta, workspace, stream=None):
    """Rotary embedding of q and k rows in place, row r of sequence b at idx[b, r]."""
    _check(lib().ec_rope(*_rope_args(q, k, idx, count, seq_len, theta, workspace),
                         _stream(stream)), "ec_rope")


LINEAR_STORE, LINEAR_RESIDUAL, LINEAR_SWIGLU = 0, 1, 2


def _linear_args(x, count, w, mode, residual, y, workspace):
    for name, t in (("x", x), ("w", w), ("y", y)):
        _cuda(name, t, torch.bfloat16)
    if mode == LINEAR_RESIDUAL:
        _cuda("residual", residual, torch.bfloat16)
    _cuda("workspace", workspace, torch.uint8)
    if count is not None:
        _cuda("count", count, torch.int32)
    if x.dim() != 3 or w.dim() != 2 or w.shape[1] != x.shape[2]:
        raise ValueError("x [batch, r_max, in], w [out (x2 for SwiGLU), in]")
    batch, r_max, n_in = x.shape
    if mode == LINEAR_SWIGLU and w.shape[0] % 2:
        raise ValueError("a SwiGLU weight stacks gate and up rows: [2 * out, in]")
    n_out = w.shape[0] // 2 if mode == LINEAR_SWIGLU else w.shape[0]
    if y.shape != (batch, r_max, n_out) or (mode == LINEAR_RESIDUAL and residual.shape != y.shape):
        raise ValueError("y (and residual) [batch, r_max, out]")
    return [_p(x), _p(count), batch, r_max, n_in, _p(w), n_out, int(mode),
            _p(residual) if mode == LINEAR_RESIDUAL else None, _p(y), _p(workspace),
            workspace.numel()]


def ec_linear(x, count, w, mode, residual, y, workspace, stream=None):
    """y = x w^T (mode 0), residual + x w^T (1), silu(x w_g^T) * x w_u^T (2, w = [w_g; w_u])."""
    _check(lib().ec_linear(*_linear_args(x, count, w, mode, residual, y, workspace),
                           _stream(stream)), "ec_linear")


# ---------------------------------------------------------------------------
# Prepared calls: validate and marshal once, then invoke with almost no host
# cost.  The tensors bound at preparation must stay alive and in place.


class Prepared:
    """A C-ABI call whose arguments are already validated and converted.  It holds
    raw device pointers, so it also keeps a reference to every object it was
    prepared from (``keep``): the tensors cannot be freed while the call lives."""

    def __init__(self, name, args, stream, keep=()):
        self.name = name
        self._keep = tuple(keep)
        self.fn = getattr(lib(), name)
        args = list(args) + [_stream(stream)]
        # pre-convert every argument to its ctypes type so a call converts nothing
        self.args = [a if (a is None or isinstance(a, t)) else t(a)
                     for a, t in zip(args, self.fn.argtypes)]

    def set_arg(self, i, value):
        t = self.fn.argtypes[i]
        self.args[i] = value if isinstance(value, t) else t(value)

    def __call__(self):
        rc = self.fn(*self.args)
        if rc != 0:
            raise ECError(rc, self.name)


def prepare_decode_step(*args, stream=None, **kwargs):
    """ec_decode_step bound to fixed buffers; ``.set_step(t)`` changes the step index."""
    p = Prepared("ec_decode_step", _decode_args(*args, **kwargs), stream,
                 keep=(args, kwargs))
    p.set_step = lambda t: p.set_arg(11, int(t))
    return p


def prepare_lmhead_decode_step(*args, stream=None, **kwargs):
    return Prepared("ec_lmhead_decode_step", _lmhead_args(*args, **kwargs), stream,
                    keep=(args, kwargs))


def prepare_build_recompute_set(*args, stream=None, **kwargs):
    return Prepared("ec_build_recompute_set", _recompute_args(*args, **kwargs), stream,
                    keep=(args, kwargs))


def prepare_selective_attention(*args, stream=None, **kwargs):
    return Prepared("ec_selective_attention", _attention_args(*args, **kwargs), stream,
                    keep=(args, kwargs))


def prepare_cover_seed_score(*args, stream=None, **kwargs):
    return Prepared("ec_cover_seed_score", _cover_score_args(*args, **kwargs), stream,
                    keep=(args, kwargs))


def prepare_selective_attention_simsd(*args, stream=None, **kwargs):
    return Prepared("ec_selective_attention_simsd", _simsd_args(*args, **kwargs), stream,
                    keep=(args, kwargs))


def prepare_selective_attention_cover(*args, stream=None, **kwargs):
    return Prepared("ec_selective_attention_cover", _cover_args(*args, **kwargs), stream,
                    keep=(args, kwargs))


def prepare_rms_norm(*args, stream=None, **kwargs):
    return Prepared("ec_rms_norm", _rms_norm_args(*args, **kwargs), stream, keep=(args, kwargs))


def prepare_rope(*args, stream=None, **kwargs):
    return Prepared("ec_rope", _rope_args(*args, **kwargs), stream, keep=(args, kwargs))


def prepare_linear(*args, stream=None, **kwargs):
    return Prepared("ec_linear", _linear_args(*args, **kwargs), stream, keep=(args, kwargs))


def prepare_embed_rows(*args, stream=None, **kwargs):
    return Prepared("ec_embed_rows", _embed_args(*args, **kwargs), stream,
                    keep=(args, kwargs))


def prepare_qkv_projection(*args, stream=None, **kwargs):
    return Prepared("ec_qkv_projection", _projection_args(*args, **kwargs), stream,
                    keep=(args, kwargs))
