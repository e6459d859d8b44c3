"""ctypes wrapper of the float64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this module.  The CUDA library and its
Python binding never do, and this module never imports them.

Every function takes numpy arrays (host memory) and returns numpy arrays; the
arithmetic is all in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

F32, BF16, F64 = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with plain ``-O2`` (no fast-math) and OpenMP over
    independent items, if stale."""
    if force or not os.path.exists(LIBRARY) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-fopenmp", "-shared",
                               "-o", LIBRARY, SOURCE, "-lm"])
    return LIBRARY


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIBRARY)
        vp, i32, i64, f32, f64 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_float, ctypes.c_double)
        L.orc_row_stats.argtypes = [vp, ctypes.c_int, i64, i32, i32, vp, vp, vp]
        L.orc_unmask_gate.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, f32, i32,
                                      vp, vp, vp, vp, vp, vp]
        L.orc_recompute_set.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]
        L.orc_scatter_kv.argtypes = [vp, vp, ctypes.c_int, vp, i64, vp, vp, vp,
                                     i32, i32, i32, i32, i32]
        L.orc_attention.argtypes = [vp, vp, vp, ctypes.c_int, vp, i32, i32, i32, i32, i32, i32,
                                    f64, vp, i64, vp]
        L.orc_attention_simsd.argtypes = [vp, vp, vp, ctypes.c_int, vp, i64, vp, vp, vp, i32, i32,
                                          i32, i32, i32, i32, f64, vp, i64, vp]
        L.orc_attention_cover.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, vp, i64, vp, vp, i32,
                                          i32, i32, i32, i32, i32, f64, vp]
        L.orc_cover_seed_score.argtypes = [vp, vp, ctypes.c_int, vp, i64, vp, vp, vp, vp, i32, i32,
                                           i32, i32, i32, i32, f64, i32, vp, vp, vp, vp]
        L.orc_embed_rows.argtypes = [vp, ctypes.c_int, i64, i32, vp, i64, vp, vp, vp, i32, i32,
                                     i32, i32, vp]
        L.orc_projection.argtypes = [vp, vp, ctypes.c_int, i64, i32, i32, vp, i64, vp]
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_set_threads.restype = None
        L.orc_get_threads.argtypes = []
        L.orc_get_threads.restype = ctypes.c_int
        for fn in (L.orc_row_stats, L.orc_unmask_gate, L.orc_recompute_set,
                   L.orc_scatter_kv, L.orc_attention, L.orc_attention_simsd,
                   L.orc_attention_cover, L.orc_embed_rows, L.orc_projection):
            fn.restype = ctypes.c_int
        _lib = L
    return _lib


def set_threads(n: int) -> None:
    """Host threads for the loops over independent rows / outputs (default 1).
    Every item is computed by one thread, so results do not depend on n."""
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return lib().orc_get_threads()


def usable_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def _dtype_of(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"oracle takes float32, bf16 bits (uint16) or float64, got {a.dtype}")


def row_stats(logits: np.ndarray):
    """(entropy f64[N], conf f64[N], token i32[N]) of each row of ``[N, V]`` logits."""
    x = np.ascontiguousarray(logits)
    n, v = x.shape
    h = np.empty(n, np.float64)
    c = np.empty(n, np.float64)
    t = np.empty(n, np.int32)
    _check(lib().orc_row_stats(_p(x), _dtype_of(x), v, n, v, _p(h), _p(c), _p(t)), "row_stats")
    return h, c, t


def unmask_gate(conf, entropy, token, seq_row_offsets, row_pos, seq_len, n_unmask, tau, step,
                is_masked, tokens, decode_step):
    """Unmask, max entropy and gate for one step.  The three state arrays are
    copied, updated and returned; the inputs are left unchanged."""
    conf = np.ascontiguousarray(conf, np.float64)
    entropy = np.ascontiguousarray(entropy, np.float64)
    token = np.ascontiguousarray(token, np.int32)
    off = np.ascontiguousarray(seq_row_offsets, np.int32)
    pos = np.ascontiguousarray(row_pos, np.int32)
    batch = off.shape[0] - 1
    im = np.array(is_masked, np.uint8, copy=True, order="C")
    tk = np.array(tokens, np.int32, copy=True, order="C")
    ds = np.array(decode_step, np.int32, copy=True, order="C")
    unmask = np.empty(batch * n_unmask, np.int32)
    e = np.empty(batch, np.float64)
    refresh = np.empty(batch, np.uint8)
    _check(lib().orc_unmask_gate(_p(conf), _p(entropy), _p(token), _p(off), _p(pos), batch,
                                 seq_len, n_unmask, float(np.float32(tau)), step, _p(unmask),
                                 _p(e), _p(refresh), _p(im), _p(tk), _p(ds)), "unmask_gate")
    return dict(unmask_rows=unmask.reshape(batch, n_unmask), max_entropy=e, refresh=refresh,
                is_masked=im, tokens=tk, decode_step=ds)


def recompute_set(is_masked, decode_step, refresh, block_lo, block_hi, k):
    """(idx i32[B, L] ascending and -1 padded, count i32[B])."""
    im = np.ascontiguousarray(is_masked, np.uint8)
    ds = np.ascontiguousarray(decode_step, np.int32)
    rf = np.ascontiguousarray(refresh, np.uint8)
    batch, seq_len = im.shape
    idx = np.empty((batch, seq_len), np.int32)
    cnt = np.empty(batch, np.int32)
    _check(lib().orc_recompute_set(_p(im), _p(ds), _p(rf), batch, seq_len, block_lo, block_hi,
                                   k, _p(idx), _p(cnt)), "recompute_set")
    return idx, cnt


def scatter_kv(k_new, v_new, idx, count, k_cache, v_cache):
    """Copies of the caches with the fresh rows written at ``idx``."""
    kn = np.ascontiguousarray(k_new)
    vn = np.ascontiguousarray(v_new)
    kc = np.array(k_cache, copy=True, order="C")
    vc = np.array(v_cache, copy=True, order="C")
    ix = np.ascontiguousarray(idx, np.int32)
    cnt = np.ascontiguousarray(count, np.int32)
    batch, seq_len, hkv, d = kc.shape
    r_max = kn.shape[1]
    dt = _dtype_of(kc)
    if not (_dtype_of(kn) == _dtype_of(vn) == _dtype_of(vc) == dt):
        raise TypeError("mixed dtypes")
    _check(lib().orc_scatter_kv(_p(kn), _p(vn), dt, _p(ix), ix.shape[-1], _p(cnt), _p(kc),
                                _p(vc), batch, seq_len, r_max, hkv, d), "scatter_kv")
    return kc, vc


def attention(q, k_cache, v_cache, count, scale, samples=None):
    """float64 attention outputs.  ``samples`` None: ``[B, r_max, H, d]`` with rows
    past ``count`` set to NaN; else an ``[S, 3]`` array of (b, r, h) and the result
    is ``[S, d]``."""
    qq = np.ascontiguousarray(q)
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    cnt = np.ascontiguousarray(count, np.int32)
    batch, r_max, h, d = qq.shape
    seq_len, hkv = kc.shape[1], kc.shape[2]
    dt = _dtype_of(qq)
    if samples is None:
        out = np.full((batch, r_max, h, d), np.nan, np.float64)
        sp, ns = None, 0
    else:
        sp = np.ascontiguousarray(samples, np.int32).reshape(-1, 3)
        ns = sp.shape[0]
        out = np.empty((ns, d), np.float64)
    _check(lib().orc_attention(_p(qq), _p(kc), _p(vc), dt, _p(cnt), batch, seq_len, r_max, h,
                               hkv, d, float(scale), _p(sp), ns, _p(out)), "attention")
    return out


def attention_simsd(q, k_cache, v_cache, idx, count, section, tau, scale, samples=None):
    """float64 attention under SimSD's temporal causal mask (``oracle.c``,
    ``orc_attention_simsd``).  ``idx`` [B, >= r_max] gives each query row's
    position, ``section`` uint8 and ``tau`` int32 [B, L] the layout.  Same output
    shapes as :func:`attention`."""
    qq = np.ascontiguousarray(q)
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    ix = np.ascontiguousarray(idx, np.int32)
    cnt = np.ascontiguousarray(count, np.int32)
    sec = np.ascontiguousarray(section, np.uint8)
    tl = np.ascontiguousarray(tau, np.int32)
    batch, r_max, h, d = qq.shape
    seq_len, hkv = kc.shape[1], kc.shape[2]
    assert sec.shape == (batch, seq_len) and tl.shape == (batch, seq_len)
    dt = _dtype_of(qq)
    if samples is None:
        out = np.full((batch, r_max, h, d), np.nan, np.float64)
        sp, ns = None, 0
    else:
        sp = np.ascontiguousarray(samples, np.int32).reshape(-1, 3)
        ns = sp.shape[0]
        out = np.empty((ns, d), np.float64)
    _check(lib().orc_attention_simsd(_p(qq), _p(kc), _p(vc), dt, _p(ix), ix.shape[-1], _p(cnt),
                                     _p(sec), _p(tl), batch, seq_len, r_max, h, hkv, d,
                                     float(scale), _p(sp), ns, _p(out)), "attention_simsd")
    return out


def attention_cover(q, k_new, v_new, k_cache, v_cache, idx, count, seed, scale):
    """COVER's dual-view attention (``oracle.c``, ``orc_attention_cover``):
    returns ``(k_cache', v_cache', out)``: the caches after the write-back of the
    non-seed rows and the float64 outputs ``[B, r_max, H, d]`` (rows past count
    NaN).  ``seed`` uint8 ``[B, r_max]`` flags the recomputed rows that are seeds."""
    qq = np.ascontiguousarray(q)
    kn = np.ascontiguousarray(k_new)
    vn = np.ascontiguousarray(v_new)
    kc = np.array(k_cache, copy=True, order="C")
    vc = np.array(v_cache, copy=True, order="C")
    ix = np.ascontiguousarray(idx, np.int32)
    cnt = np.ascontiguousarray(count, np.int32)
    sd = np.ascontiguousarray(seed, np.uint8)
    batch, r_max, h, d = qq.shape
    seq_len, hkv = kc.shape[1], kc.shape[2]
    assert sd.shape == (batch, r_max)
    dt = _dtype_of(qq)
    out = np.empty((batch, r_max, h, d), np.float64)
    _check(lib().orc_attention_cover(_p(qq), _p(kn), _p(vn), _p(kc), _p(vc), dt, _p(ix),
                                     ix.shape[-1], _p(cnt), _p(sd), batch, seq_len, r_max, h, hkv,
                                     d, float(scale), _p(out)), "attention_cover")
    return kc, vc, out


def cover_seed_score(q, k_cache, idx, count, role, drafted, u, scale, n_seed):
    """COVER's seed score (``oracle.c``, ``orc_cover_seed_score``): returns
    ``(d_in, d_out, score, seeds)``; the first three float64 ``[B, r_max]``, NaN
    except at candidate rows, ``seeds`` int32 ``[B, n_seed]`` positions (-1 pad).
    ``role`` uint8 ``[B, r_max]`` (bit 0 still masked, bit 1 candidate),
    ``drafted`` uint8 ``[B, L]``, ``u`` ``[B, r_max]`` (widened to float64)."""
    qq = np.ascontiguousarray(q)
    kc = np.ascontiguousarray(k_cache)
    ix = np.ascontiguousarray(idx, np.int32)
    cnt = np.ascontiguousarray(count, np.int32)
    rl = np.ascontiguousarray(role, np.uint8)
    dr = np.ascontiguousarray(drafted, np.uint8)
    uu = np.ascontiguousarray(u, np.float64)
    batch, r_max, h, d = qq.shape
    seq_len, hkv = kc.shape[1], kc.shape[2]
    assert rl.shape == (batch, r_max) and uu.shape == (batch, r_max)
    assert dr.shape == (batch, seq_len) and kc.dtype == qq.dtype
    dt = _dtype_of(qq)
    d_in, d_out, score = (np.empty((batch, r_max), np.float64) for _ in range(3))
    seeds = np.empty((batch, n_seed), np.int32)
    _check(lib().orc_cover_seed_score(_p(qq), _p(kc), dt, _p(ix), ix.shape[-1], _p(cnt), _p(rl),
                                      _p(dr), _p(uu), batch, seq_len, r_max, h, hkv, d,
                                      float(scale), n_seed, _p(d_in), _p(d_out), _p(score),
                                      _p(seeds)), "cover_seed_score")
    return d_in, d_out, score, seeds


def embed_rows(table, idx, count, tokens, is_masked, mask_id, r_max):
    """``[B, r_max, hidden]`` rows of ``table`` for the recomputed positions; rows
    past ``count`` are zero."""
    tb = np.ascontiguousarray(table)
    ix = np.ascontiguousarray(idx, np.int32)
    cnt = np.ascontiguousarray(count, np.int32)
    tk = np.ascontiguousarray(tokens, np.int32)
    im = np.ascontiguousarray(is_masked, np.uint8)
    batch, seq_len = tk.shape
    rows, hidden = tb.shape
    x = np.zeros((batch, r_max, hidden), tb.dtype)
    _check(lib().orc_embed_rows(_p(tb), _dtype_of(tb), rows, hidden, _p(ix), ix.shape[-1], _p(cnt),
                                _p(tk), _p(im), int(mask_id), batch, seq_len, r_max, _p(x)),
           "embed_rows")
    return x


def projection(x, w, rows=None):
    """float64 ``x @ w.T`` for ``x [n, hidden]``, ``w [n_out, hidden]`` (same element
    type); with ``rows`` only those rows of x, in that order."""
    xx = np.ascontiguousarray(x)
    ww = np.ascontiguousarray(w)
    if _dtype_of(xx) != _dtype_of(ww):
        raise TypeError("mixed dtypes")
    n, hidden = xx.shape
    n_out = ww.shape[0]
    if ww.shape[1] != hidden:
        raise ValueError("inner dimensions differ")
    if rows is None:
        sel, ns = None, 0
        y = np.empty((n, n_out), np.float64)
    else:
        sel = np.ascontiguousarray(rows, np.int64)
        ns = sel.shape[0]
        y = np.empty((ns, n_out), np.float64)
    _check(lib().orc_projection(_p(xx), _p(ww), _dtype_of(xx), n, hidden, n_out, _p(sel), ns,
                                _p(y)), "projection")
    return y
