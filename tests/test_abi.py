"""The C ABI library loads without a GPU, exports every entry point declared in
include/ec.h, and rejects bad arguments on the host before launching anything."""
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
    text = open(os.path.join(ROOT, "include", "ec.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ec_[a-z_]+)\s*\(", text)))


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
