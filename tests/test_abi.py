"""The C ABI library loads without a GPU, exports every entry point declared in
include/*.h, and rejects bad arguments on the host before launching anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from entropy_gated_kv_decode_b300 import build, _native
    build.build()
    return _native.lib()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for h in sorted(os.listdir(inc)):
        if h.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, h)).read(), flags=re.S)
            names |= set(re.findall(r"\b(ec_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    from entropy_gated_kv_decode_b300 import _native
    assert sorted(_native.EXPORTED) == names


def test_status_strings_and_version(L):
    assert L.ec_abi_version() == 1
    for code in range(0, -8, -1):
        s = L.ec_status_str(code).decode()
        assert s.startswith("EC_")
    assert "unknown" in L.ec_status_str(42).decode()


def test_workspace_sizes(L):
    small = L.ec_decode_workspace_size(32, 1)
    big = L.ec_decode_workspace_size(512, 8)
    assert small >= 256 and big > small and big % 16 == 0
    assert L.ec_attention_workspace_size(8, 2048, 96, 28, 4, 128) >= 256


def _decode(L, **over):
    a = dict(logits=0x1000, dtype=1, row_stride=126464, n_rows=32, vocab=126464, offsets=0x2000,
             row_pos=0x3000, batch=1, seq_len=1024, n_unmask=2, tau=0.5, step=0, tok=0x4000,
             conf=0x5000, ent=0x6000, unmask=0x7000, emax=0x8000, refresh=0x9000, masked=0xa000,
             tokens=0xb000, dstep=0xc000, ws=0x10000, ws_bytes=1 << 20, stream=None)
    a.update(over)
    return L.ec_decode_step(a["logits"], a["dtype"], a["row_stride"], a["n_rows"], a["vocab"],
                            a["offsets"], a["row_pos"], a["batch"], a["seq_len"], a["n_unmask"],
                            a["tau"], a["step"], a["tok"], a["conf"], a["ent"], a["unmask"],
                            a["emax"], a["refresh"], a["masked"], a["tokens"], a["dstep"], a["ws"],
                            a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(dtype=7), -3),
    (dict(vocab=0), -2),
    (dict(n_unmask=0), -2),
    (dict(n_unmask=5000), -2),
    (dict(row_stride=100), -2),
    (dict(tau=float("nan")), -2),
    (dict(batch=0), -2),
    (dict(offsets=None), -1),
    (dict(logits=None), -1),
    (dict(ws=None), -1),
    (dict(logits=0x1008), -4),
    (dict(row_stride=126465), -4),
    (dict(ws=0x10010), -5),
    (dict(ws_bytes=100), -5),
])
def test_decode_step_rejects_bad_arguments_on_the_host(L, over, code):
    # the fake device addresses are never dereferenced: validation fails first
    assert _decode(L, **over) == code


def test_recompute_set_and_attention_reject_bad_arguments(L):
    f = L.ec_build_recompute_set
    assert f(None, 1, 1, 1, 8, 0, 4, 2, 1, 1, None) == -1
    assert f(0x100, 0x200, 0x300, 1, 8, 5, 4, 2, 0x400, 0x500, None) == -2
    assert f(0x100, 0x200, 0x300, 1, 8, 0, 9, 2, 0x400, 0x500, None) == -2
    assert f(0x100, 0x200, 0x300, 1, 8, 0, 4, -1, 0x400, 0x500, None) == -2
    g = L.ec_selective_attention
    base = [0x1000, 0x2000, 0x3000, 0x4000, 48, 0x5000, 0x6000, 0x7000, 0x8000, 1,
            1, 1024, 48, 32, 32, 128, 0.088, 0x10000, 1 << 16, None]

    def call(**kw):
        args = list(base)
        names = ["q", "kn", "vn", "idx", "stride", "count", "kc", "vc", "out", "dtype", "batch",
                 "L", "r", "H", "Hkv", "d", "scale", "ws", "wsb", "stream"]
        for k, v in kw.items():
            args[names.index(k)] = v
        return g(*args)

    assert call(d=96) == -2
    assert call(H=30, Hkv=4) == -2
    assert call(stride=40) == -2
    assert call(dtype=3) == -3
    assert call(kc=None) == -1
    assert call(q=0x1004) == -4
    assert call(ws=0x10040) == -5
    assert call(wsb=8) == -5

    # the SimSD variant: the same checks, its two label arrays, and bf16 only
    m = L.ec_selective_attention_simsd

    def call_m(**kw):
        args = list(base)
        names = ["q", "kn", "vn", "idx", "stride", "count", "kc", "vc", "out", "dtype", "batch",
                 "L", "r", "H", "Hkv", "d", "scale", "ws", "wsb", "stream"]
        for k, v in kw.items():
            if k in names:
                args[names.index(k)] = v
        sec, tau = kw.get("section", 0x20000), kw.get("tau", 0x30000)
        return m(*args[:6], sec, tau, *args[6:])

    assert call_m(d=96) == -2
    assert call_m(stride=40) == -2
    assert call_m(dtype=3) == -3
    assert call_m(section=None) == -1
    assert call_m(tau=None) == -1
    assert call_m(kc=None) == -1
    assert call_m(dtype=0) == -7  # float32: not implemented for the masked variant
    assert call_m(q=0x1004) == -4
    assert call_m(wsb=8) == -5

    # the COVER variant: its seed flags, and bf16 only
    cv = L.ec_selective_attention_cover

    def call_c(**kw):
        args = list(base)
        names = ["q", "kn", "vn", "idx", "stride", "count", "kc", "vc", "out", "dtype", "batch",
                 "L", "r", "H", "Hkv", "d", "scale", "ws", "wsb", "stream"]
        for k, v in kw.items():
            if k in names:
                args[names.index(k)] = v
        return cv(*args[:6], kw.get("seed", 0x20000), *args[6:])

    assert call_c(d=96) == -2
    assert call_c(stride=40) == -2
    assert call_c(dtype=3) == -3
    assert call_c(seed=None) == -1
    assert call_c(kc=None) == -1
    assert call_c(dtype=0) == -7
    assert call_c(out=0x8004) == -4
    assert call_c(wsb=8) == -5


def test_projection_and_gather_reject_bad_arguments(L):
    p = L.ec_qkv_projection
    #       x       count   B  R   hidden  w       width  q       k       v       ws       wsb
    base = [0x1000, 0x2000, 1, 48, 4096, 0x3000, 12288, 0x4000, 0x5000, 0x6000, 0x10000, 256, None]

    def proj(i, v):
        args = list(base)
        args[i] = v
        return p(*args)

    assert proj(4, 4100) == -2     # hidden not a multiple of the 64-wide K step
    assert proj(6, 12290) == -2    # width not a multiple of 64
    assert proj(2, 0) == -2        # no sequences
    assert proj(10, None) == -1    # no workspace
    assert proj(0, None) == -1     # no X with rows to project
    assert proj(0, 0x1008) == -4   # X not 16-byte aligned
    assert proj(10, 0x10010) == -5  # workspace not aligned
    assert proj(11, 16) == -5      # workspace below the status header

    e = L.ec_embed_rows
    #       table   rows    hidden idx     stride count   tokens  masked  mask_id B  L     R   x       ws       wsb
    base = [0x1000, 126465, 4096, 0x2000, 48, 0x3000, 0x4000, 0x5000, 126464, 1, 1024, 48, 0x6000, 0x10000, 256, None]

    def emb(i, v):
        args = list(base)
        args[i] = v
        return e(*args)

    assert emb(2, 12) == -2        # hidden not a multiple of 8
    assert emb(8, 126465) == -2    # mask id outside the table
    assert emb(4, 40) == -2        # index stride below r_max
    assert emb(5, None) == -1      # no counts
    assert emb(0, None) == -1      # no table with rows to gather
    assert emb(12, 0x6008) == -4   # X not 16-byte aligned
    assert emb(14, 8) == -5        # workspace below the status header


def test_noalloc_decode_rejects_bad_arguments(L):
    f = L.ec_decode_step_noalloc
    #       logits  dt row_stride n_rows vocab   offsets row_pos B  L     n  tau  step tok     conf    ent     unmask  emax    refresh masked  tokens  dstep   stream
    base = [0x1000, 1, 126464,    32,    126464, 0x2000, 0x3000, 1, 1024, 2, 0.5, 0,   0x4000, 0x5000, 0x6000, 0x7000, 0x8000, 0x9000, 0xa000, 0xb000, 0xc000, None]

    def call(i, v):
        args = list(base)
        args[i] = v
        return f(*args)

    assert call(1, 7) == -3           # dtype
    assert call(4, 0) == -2           # vocab
    assert call(9, 0) == -2           # n_unmask
    assert call(2, 100) == -2         # row stride below vocab
    assert call(5, None) == -1        # offsets
    assert call(0, None) == -1        # logits with rows
    assert call(0, 0x1008) == -4      # logits not 16-byte aligned
    # a request whose scratch exceeds the fixed 2 MiB array (checked before any CUDA call)
    assert call(3, 1 << 20) == -8     # EC_ERR_SCRATCH_LIMIT


def test_noalloc_status_reader_rejects_null(L):
    assert L.ec_decode_noalloc_read_status(None, None) == -1


def test_lmhead_rejects_bad_arguments(L):
    f = L.ec_lmhead_decode_step
    #       hidden  w_lm    N    hid   V       offsets row_pos B  L     n  tau  step tok     conf    ent     unmask  emax    refresh masked  tokens  dstep   ws      ws_bytes stream
    base = [0x1000, 0x2000, 32, 4096, 126464, 0x3000, 0x4000, 1, 1024, 2, 0.5, 0,   0x5000, 0x6000, 0x7000, 0x8000, 0x9000, 0xa000, 0xb000, 0xc000, 0xd000, 0x10000, 1 << 24, None]

    def call(i, v):
        args = list(base)
        args[i] = v
        return f(*args)

    assert call(3, 100) == -2         # hidden size not a multiple of 64
    assert call(3, 0) == -2
    assert call(4, 0) == -2           # vocab
    assert call(2, 148 * 128 + 1) == -2  # more rows than 128 per SM
    assert call(9, 0) == -2           # n_unmask
    assert call(10, float("nan")) == -2  # tau
    assert call(5, None) == -1        # offsets
    assert call(0, None) == -1        # hidden with rows
    assert call(21, None) == -1       # workspace
    assert call(0, 0x1008) == -4      # hidden not 16-byte aligned
    assert call(1, 0x2004) == -4      # w_lm not 16-byte aligned
    assert call(22, 64) == -5         # workspace too small
    assert call(21, 0x10010) == -5    # workspace misaligned


def test_layer_calls_reject_bad_arguments(L):
    # ec_rms_norm(x, count, B, R, hidden, weight, eps, y, ws, wsb, stream)
    n = L.ec_rms_norm
    base = [0x1000, None, 1, 4, 4096, 0x2000, 1e-5, 0x3000, 0x10000, 256, None]

    def norm(**kw):
        names = ["x", "count", "B", "R", "hidden", "g", "eps", "y", "ws", "wsb", "stream"]
        a = list(base)
        for k, v in kw.items():
            a[names.index(k)] = v
        return n(*a)

    assert norm(hidden=12) == -2
    assert norm(eps=-1.0) == -2
    assert norm(eps=float("nan")) == -2
    assert norm(x=None) == -1
    assert norm(g=0x2004) == -4
    assert norm(wsb=4) == -5
    # ec_rope(q, k, idx, stride, count, B, L, R, H, Hkv, d, theta, ws, wsb, stream)
    r = L.ec_rope
    rb = [0x1000, 0x2000, 0x3000, 8, 0x4000, 1, 1024, 8, 4, 2, 128, 10000.0, 0x10000, 256, None]

    def rope(**kw):
        names = ["q", "k", "idx", "stride", "count", "B", "L", "R", "H", "Hkv", "d", "theta", "ws",
                 "wsb", "stream"]
        a = list(rb)
        for key, v in kw.items():
            a[names.index(key)] = v
        return r(*a)

    assert rope(d=129) == -2
    assert rope(d=256) == -2
    assert rope(theta=1.0) == -2
    assert rope(stride=4) == -2
    assert rope(count=None) == -1
    assert rope(q=None) == -1
    # ec_linear(x, count, B, R, in, w, out, mode, residual, y, ws, wsb, stream)
    f = L.ec_linear
    lb = [0x1000, None, 1, 4, 4096, 0x2000, 4096, 0, None, 0x3000, 0x10000, 256, None]

    def lin(**kw):
        names = ["x", "count", "B", "R", "in", "w", "out", "mode", "res", "y", "ws", "wsb", "stream"]
        a = list(lb)
        for key, v in kw.items():
            a[names.index(key)] = v
        return f(*a)

    assert lin(mode=3) == -2
    assert lin(**{"in": 100}) == -2
    assert lin(out=96) == -2             # a plain output is a multiple of 64
    assert lin(mode=2, out=96, w=0x2008) == -4  # SwiGLU: a multiple of 32 passes the shape check ...
    assert lin(mode=2, out=48) == -2      # ... and at least 64
    assert lin(mode=1) == -1              # the residual form needs its residual
    assert lin(w=0x2008) == -4
    assert lin(wsb=4) == -5


def test_cover_seed_score_rejects_bad_arguments_on_the_host(L):
    # every case below fails validation, so the fake device addresses are never used
    f = L.ec_cover_seed_score
    names = ["q", "k", "idx", "stride", "count", "role", "drafted", "u", "dtype", "B", "L", "R", "H",
             "Hkv", "d", "scale", "n_seed", "d_in", "d_out", "score", "seeds", "ws", "wsb", "stream"]
    base = [0x1000, 0x2000, 0x3000, 96, 0x4000, 0x5000, 0x6000, 0x7000, 1, 8, 2048, 96, 28, 4, 128,
            0.088, 8, 0x8000, 0x9000, 0xa000, 0xb000, 0x10000, 1 << 40, None]

    def call(**kw):
        a = list(base)
        for key, v in kw.items():
            a[names.index(key)] = v
        return f(*a)

    assert call(dtype=7) == -3
    assert call(dtype=0) == -7             # float32 is not implemented
    assert call(d=96) == -7
    assert call(B=0) == -2
    assert call(Hkv=5) == -2
    assert call(stride=95) == -2
    assert call(n_seed=-1) == -2
    assert call(scale=float("nan")) == -2
    assert call(count=None) == -1
    assert call(q=None) == -1
    assert call(drafted=None) == -1
    assert call(seeds=None) == -1          # seeds asked for
    assert call(ws=None) == -1
    assert call(q=0x1008) == -4
    assert call(k=0x2004) == -4
    assert call(ws=0x10010) == -5
    assert call(wsb=L.ec_cover_score_workspace_size(8, 2048, 96, 28) - 1) == -5
    # no rows and no seed slots: nothing to launch
    assert call(R=0, stride=0, n_seed=0, seeds=None, wsb=256) == 0


def test_cover_score_sizes_and_launches(L):
    small = L.ec_cover_score_workspace_size(1, 1024, 48, 32)
    big = L.ec_cover_score_workspace_size(8, 2048, 96, 28)
    assert small >= 256 and big > small and big % 256 == 0
    assert L.ec_cover_score_workspace_size(1, 8192, 0, 32) == 256  # the status word only
    assert L.ec_cover_score_kernel_count(8, 96, 8) == 5
    assert L.ec_cover_score_kernel_count(8, 96, 0) == 4
    assert L.ec_cover_score_kernel_count(8, 0, 4) == 1
    assert L.ec_cover_score_kernel_count(8, 0, 0) == 0
