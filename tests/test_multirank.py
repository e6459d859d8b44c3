"""The N-replica bench path on CPU: two gloo ranks run the same barrier,
max-over-ranks and whole-job throughput logic that bench.py uses under torchrun
(the path has no data exchange; ranks are independent replicas), and the
reference arm only prints on rank 0."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
args = bench.parse_args([])
rank, world, local = bench.dist_setup(args)
assert dist.get_backend() == "gloo"
bench.barrier(world)
mine = 1.0 + rank          # seconds this rank "took"
t = bench.reduce_max(mine, world)
value = bench.aggregate(100.0, world, t)
print(json.dumps({{"rank": rank, "world": world, "max": t, "value": value}}), flush=True)
dist.destroy_process_group()
"""


def _run_ranks(code, world=2, extra_env=None):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_two_gloo_ranks_take_the_slowest_rank_time():
    outs = _run_ranks(WORKER.format(root=ROOT))
    lines = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    for d in lines:
        assert d["world"] == 2
        assert d["max"] == 2.0                       # the slower rank's time
        assert d["value"] == pytest.approx(100.0)    # 2 ranks x 100 units / 2 s


def test_reference_arm_prints_only_on_rank_zero():
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
            "bench.main(['--impl', 'reference', '--workload', 'tiny', '--steps', '1', "
            "'--warmup', '0', '--cpu-seconds', '0.05'])")
    outs = _run_ranks(code)
    assert outs[1].strip() == ""
    d = json.loads(outs[0].strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
