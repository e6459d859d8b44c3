"""The attention call's work split, as the library reports it through
ec_attention_kernel_count (host logic only: without a device the library plans for
148 SMs).  A split plan launches the write-back, the attention and the merge
kernel; whole units need no merge."""
import pytest
import torch


def native():
    from entropy_gated_kv_decode_b300 import build, _native
    build.build()
    return _native


@pytest.mark.parametrize("shape,launches", [
    ((1, 1024, 48, 32, 32, 128), 3),     # single sequence: 32 units of 8 tiles, 4 splits
    ((8, 2048, 96, 28, 4, 128), 3),      # batched GQA: stream-K
    ((1, 8192, 288, 32, 32, 128), 3),    # long context: split-major items
    ((1, 1024, 1024, 32, 32, 128), 2),   # full refresh: 256 whole units
    ((1, 64, 32, 2, 2, 64), 2),          # one key tile per unit: nothing to split
    ((1, 1, 48, 32, 32, 128), 2),        # a single key
    ((1, 256, 48, 32, 32, 128), 2),      # two key tiles: too short to split
    ((4, 512, 64, 8, 8, 128), 2),        # 32 units of 4 tiles: whole units beat a split + merge
    ((1, 1024, 48, 32, 32, 64), 3),      # head_dim 64, as the single sequence
    ((2, 4096, 200, 16, 2, 128), 3),     # GQA 8:1, several row tiles per KV head
    ((1, 1024, 0, 32, 32, 128), 0),      # no recomputed rows: no launch at all
])
def test_attention_launches(shape, launches):
    nat = native()
    assert nat.ec_attention_kernel_count(torch.bfloat16, *shape) == launches
    # float32 runs the write-back and the CUDA-core kernel
    assert nat.ec_attention_kernel_count(torch.float32, *shape) == (2 if shape[2] else 0)


def test_rejected_shapes():
    nat = native()
    assert nat.ec_attention_kernel_count(torch.bfloat16, 1, 1024, 48, 32, 5, 128) == -1  # H % Hkv
    assert nat.ec_attention_kernel_count(torch.bfloat16, 1, 1024, 48, 32, 32, 96) == -1  # head_dim
    assert nat.ec_attention_kernel_count(torch.bfloat16, 0, 1024, 48, 32, 32, 128) == -1  # batch
