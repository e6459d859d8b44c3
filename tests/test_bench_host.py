"""Host-side pieces of bench.py: the packed transfer buffers and the stored
traffic figure's guard on the kernel sources."""
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_packed_views_are_aligned_disjoint_and_contiguous():
    specs = [("logits", (3, 7), torch.bfloat16), ("q", (2, 5, 4), torch.float32),
             ("flag", (3,), torch.uint8), ("idx", (2, 9), torch.int32)]
    p = bench.Packed(specs, "cpu")
    assert all(o % 256 == 0 for o in p.offsets) and p.nbytes % 256 == 0
    for (name, shape, dtype), o in zip(specs, p.offsets):
        v = p.views[name]
        assert v.shape == shape and v.dtype == dtype and v.is_contiguous()
        assert v.data_ptr() - p.blob.data_ptr() == o
    # writing one view leaves the others untouched
    p.blob.zero_()
    p.views["q"].fill_(1.5)
    assert not p.views["logits"].any() and not p.views["flag"].any() and not p.views["idx"].any()
    # one blob copy moves every view
    q = bench.Packed(specs, "cpu")
    q.blob.copy_(p.blob)
    assert torch.equal(q.views["q"], p.views["q"])


def test_traffic_is_reported_only_for_the_captured_sources():
    h = bench.kernel_sources_hash(files=bench.CALL_SOURCES["attention"])
    assert len(h) == 16 and int(h, 16) >= 0
    saved = dict(bench.MEASURED_TRAFFIC)
    try:
        bench.MEASURED_TRAFFIC.clear()
        bench.MEASURED_TRAFFIC[("w", "attention")] = {"sources": h, "bytes": 123}
        bench.MEASURED_TRAFFIC[("w", "decode")] = {"sources": "0" * 16, "bytes": 456}
        assert bench.measured_traffic("w", "attention") == 123
        assert bench.measured_traffic("w", "decode") is None      # kernels changed since
        assert bench.measured_traffic("other", "attention") is None
    finally:
        bench.MEASURED_TRAFFIC.clear()
        bench.MEASURED_TRAFFIC.update(saved)


def test_call_hash_covers_its_own_files_only(tmp_path):
    a, b = tmp_path / "a.cu", tmp_path / "b.cu"
    a.write_text("__global__ void ka(int *p) { p[0] = 1; }\n")
    b.write_text("__global__ void kb(int *p) { p[0] = 1; }\n")
    h0 = bench.kernel_sources_hash(files=[str(a)])
    b.write_text("__global__ void kb(int *p) { p[0] = 2; }\n")
    assert bench.kernel_sources_hash(files=[str(a)]) == h0  # another call's kernel changed
    a.write_text("__global__ void ka(int *p) { p[0] = 3; }\n")
    assert bench.kernel_sources_hash(files=[str(a)]) != h0
    for call, files in bench.CALL_SOURCES.items():  # every listed file exists
        assert bench.kernel_sources_hash(files=files)


def test_sources_hash_ignores_comments_but_not_code(tmp_path):
    src = tmp_path / "k.cu"
    src.write_text('// a kernel\n__global__ void k(int *p) { p[0] = 1; /* one */ }\n'
                   'const char *s = "// not a comment";\n')
    h0 = bench.kernel_sources_hash(str(tmp_path))
    src.write_text('// the kernel, reworded\n__global__ void k(int *p)\n{\n    p[0] = 1;\n}\n'
                   'const char *s = "// not a comment";\n')
    assert bench.kernel_sources_hash(str(tmp_path)) == h0
    src.write_text('// a kernel\n__global__ void k(int *p) { p[0] = 2; }\n'
                   'const char *s = "// not a comment";\n')
    assert bench.kernel_sources_hash(str(tmp_path)) != h0
    src.write_text('// a kernel\n__global__ void k(int *p) { p[0] = 1; }\n'
                   'const char *s = "// not a comment!";\n')
    assert bench.kernel_sources_hash(str(tmp_path)) != h0  # string contents are code
