"""The attention call's launches and workspace, as the library reports them
through ec_attention_kernel_count and ec_attention_workspace_size (host logic
only: without a device the library plans for 148 SMs).  The bf16 tensor-core
path is one kernel whatever the split (the KV write-back and the merge of split
units run inside it); float32 runs a write-back and the CUDA-core kernel."""
import pytest
import torch


def native():
    from entropy_gated_kv_decode_b300 import build, _native
    build.build()
    return _native


SHAPES = [
    (1, 1024, 48, 32, 32, 128),     # single sequence: 32 units of 8 tiles
    (8, 2048, 96, 28, 4, 128),      # batched GQA: groups of 6 CTAs
    (1, 8192, 288, 32, 32, 128),    # long context: groups of 3 CTAs
    (1, 1024, 1024, 32, 32, 128),   # full refresh: groups of 8 CTAs
    (1, 64, 32, 2, 2, 64),          # one key tile per unit
    (1, 1, 48, 32, 32, 128),        # a single key
    (1, 256, 48, 32, 32, 128),      # two key tiles
    (4, 512, 64, 8, 8, 128),        # 32 units of 4 tiles
    (1, 1024, 48, 32, 32, 64),      # head_dim 64
    (2, 4096, 200, 16, 2, 128),     # GQA 8:1, several row tiles per KV head
    (1, 8192, 8192, 32, 32, 128),   # 64 units per head: whole units dealt round-robin
]


@pytest.mark.parametrize("shape", SHAPES)
def test_one_launch(shape):
    nat = native()
    assert nat.ec_attention_kernel_count(torch.bfloat16, *shape) == 1
    assert nat.ec_attention_kernel_count(torch.float32, *shape) == 2


def test_no_rows_no_launch():
    nat = native()
    assert nat.ec_attention_kernel_count(torch.bfloat16, 1, 1024, 0, 32, 32, 128) == 0
    assert nat.ec_attention_kernel_count(torch.float32, 1, 1024, 0, 32, 32, 128) == 0


def test_workspace_holds_the_split_partials():
    nat = native()
    header = 256
    # one tile per unit: no unit is cut, only the header and the per-unit flags
    small = nat.ec_attention_workspace_size(1, 64, 32, 2, 2, 64)
    assert header < small <= header + 256
    # batched GQA: units cut between groups keep (O, m, l) partials: at least one
    # 128-row slot of 128 floats + (m, l) per unit
    units = 8 * 4 * 6
    big = nat.ec_attention_workspace_size(8, 2048, 96, 28, 4, 128)
    assert big >= units * 128 * (128 + 2) * 4
    # 64 units per head in two groups of 64 CTAs, each covering 16 whole heads:
    # no unit is cut, so no partials
    whole = nat.ec_attention_workspace_size(1, 8192, 8192, 32, 32, 128)
    assert whole <= header + 32 * 64 * 4 + 256


def test_rejected_shapes():
    nat = native()
    assert nat.ec_attention_kernel_count(torch.bfloat16, 1, 1024, 48, 32, 5, 128) == -1  # H % Hkv
    assert nat.ec_attention_kernel_count(torch.bfloat16, 1, 1024, 48, 32, 32, 96) == -1  # head_dim
    assert nat.ec_attention_kernel_count(torch.bfloat16, 0, 1024, 48, 32, 32, 128) == -1  # batch
