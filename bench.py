#!/usr/bin/env python
"""Benchmark of the EntropyCache per-step hot path on B300.

One step = one pass of the whole hot path over one batch of synthetic input,
in the order a denoising step runs it:
  1. ec_selective_attention  — write the recomputed K/V rows into the cache and
     attend from those rows over all L cached keys (the partial forward);
  2. ec_decode_step          — entropy / confidence / token per masked row,
     confidence-ranked unmasking, max entropy E and the E > tau gate;
  3. ec_build_recompute_set  — the index set of the next forward.

Metric: entropy/gate GB/s = bytes of logits the decode-and-gate call consumes
per second of its own device time (N * V * element size / call time).  The
line also carries the whole step's time and logits rate, the attention call's
TFLOP/s and fraction of the tensor peak, and a roofline object for the
dominant call, all measured live with CUDA events on the launching stream.
Each call (and the whole step) is a CUDA graph with its own pair of events; L2
is flushed (a 256 MiB write, then a 256 MiB read) before every timed replay,
outside the timed intervals.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME|all]
                  [--impl ours|reference]

N > 1 runs under torchrun: every rank runs an independent replica (the path
has no exchange step), the timed region is bracketed by barriers, and the
slowest rank's time is used.  --impl reference times the float64 CPU oracle
on the host cores instead.  --workload all prints one line per workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from entropy_gated_kv_decode_b300 import synth  # noqa: E402

METRIC = "entropy/gate GB/s (% HBM peak); selective-recompute attention TFLOP/s (% peak)"
DEFAULT_WORKLOAD = "batched"
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

# DRAM bytes (read + write) per call of the dominant call, from one ncu capture of
# the same bench command (dram__bytes_read.sum + dram__bytes_write.sum summed over
# the call's kernels, per launch).  Used only while the files the call is built
# from (CALL_SOURCES) hash to the value they had when the counters were taken.
MEASURED_TRAFFIC = {
    # `bench.py --steps 20 --warmup 3 --e2e-steps 100 --cpu-seconds 0.1 --no-lmhead
    # --no-simsd --no-cover`, mean of two launches; the decode call is both of its kernels
    ("batched", "attention"): {"bytes": 39193728, "sources": "bfc20f966a175408"},
    ("batched", "decode"): {"bytes": 156080896, "sources": "514662fb16117650"},
}

# The files a measured call's kernels are compiled from: the kernels' own source,
# the device headers it includes, the C ABI entry that validates and launches it
# (kernel attributes are set there) and the public header.
CALL_SOURCES = {
    "decode": ("csrc/decode_gate.cu", "csrc/gate_common.cuh", "csrc/tc_ptx.cuh",
               "csrc/ec_internal.cuh", "csrc/ec_api.cu", "../include/ec.h"),
    "attention": ("csrc/attention_tc.cu", "csrc/tc_ptx.cuh", "csrc/ec_internal.cuh",
                  "csrc/ec_api.cu", "../include/ec.h"),
}


def _code_only(text: str) -> str:
    """C/C++/CUDA source without its comments and with whitespace runs collapsed:
    what the compiler sees, so that editing a comment keeps the hash."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # a string or character literal, escapes included
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_sources_hash(csrc: str | None = None, files=None) -> str:
    """Hash of kernel code, comments and layout ignored: the named files (paths
    relative to the package), else every csrc/*.cu and *.cuh of ``csrc``."""
    import hashlib
    h = hashlib.sha256()
    if files is not None:
        pkg = os.path.join(ROOT, "entropy_gated_kv_decode_b300")
        paths = [os.path.normpath(os.path.join(pkg, f)) for f in files]
    else:
        csrc = csrc or os.path.join(ROOT, "entropy_gated_kv_decode_b300", "csrc")
        paths = [os.path.join(csrc, n) for n in sorted(os.listdir(csrc)) if n.endswith((".cu", ".cuh"))]
    for path in paths:
        with open(path, encoding="utf-8") as f:
            h.update(os.path.basename(path).encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, call: str):
    t = MEASURED_TRAFFIC.get((workload, call))
    if t is None or t["sources"] != kernel_sources_hash(files=CALL_SOURCES[call]):
        return None
    return t["bytes"]


class L2Flush:
    """Evicts L2 between timed steps: writes one 256 MiB buffer, then reads a
    second one, so the next step starts with a cold L2 that holds no dirty
    lines (whose write-back would otherwise be charged to the next kernel)."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.zeros(FLUSH_BYTES // 8, dtype=torch.int64, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD,
                   choices=sorted(synth.WORKLOADS) + ["all", "lmhead"])
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--e2e-steps", type=int, default=200,
                   help="timed end-to-end steps (at least 100 are always run)")
    p.add_argument("--e2e-warmup", type=int, default=30,
                   help="untimed end-to-end steps first (at least 20 are always run)")
    p.add_argument("--eager", action="store_true", help="time eager launches, not graph replays")
    p.add_argument("--no-lmhead", action="store_true",
                   help="skip the LM-head fused decode-and-gate part")
    p.add_argument("--no-cover", action="store_true",
                   help="leave out the COVER dual-view attention part")
    p.add_argument("--no-simsd", action="store_true",
                   help="leave out the SimSD masked-attention part")
    p.add_argument("--cover-score", action="store_true",
                   help="add the COVER seed-score part (off by default)")
    p.add_argument("--cpu-seconds", type=float, default=8.0,
                   help="CPU time budget of each oracle baseline sample (one core, all cores)")
    return p.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# workload accounting (algorithmic work, independent of the implementation)


def workload_geometry(w: synth.Workload):
    elt_l = 2 if w.logits_dtype == synth.BF16 else 4
    elt_a = 2 if w.attn_dtype == synth.BF16 else 4
    r = w.r_max
    B, L, H, Hkv, d = w.batch, w.seq_len, w.n_heads, w.n_kv_heads, w.head_dim
    logits_bytes = w.n_rows * w.vocab * elt_l
    attn_flops = 4.0 * B * r * L * H * d
    attn_bytes = (2 * B * L * Hkv * d          # K and V cache read
                  + 2 * B * r * H * d          # Q read, O write
                  + 4 * B * r * Hkv * d) * elt_a  # fresh K/V read + write-back
    return dict(logits_bytes=logits_bytes, attn_flops=attn_flops, attn_bytes=attn_bytes,
                rows=w.n_rows, r=r)


def host_inputs(w: synth.Workload, seed: int):
    rng = np.random.default_rng(seed)
    st = synth.make_state(rng, w)
    logits = synth.make_logits(rng, w.n_rows, w.vocab, w.logits_dtype, w.near_uniform_frac)
    att = synth.make_attention(rng, w, w.r_max)
    return st, logits, att


# ---------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = os.path.join("/tmp", f"ec_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                if self.uuid and self.uuid not in parts[0]:
                    continue
                rows.append(parts)
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# our CUDA path


class Packed:
    """Tensors laid out in one byte buffer, each 256-byte aligned, so that a step's
    inputs (or results) move between host and device in a single copy."""

    def __init__(self, specs, device, pinned=False):
        import torch
        self.offsets, off = [], 0
        for _, shape, dtype in specs:
            self.offsets.append(off)
            n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            off += (n + 255) // 256 * 256
        self.nbytes = off
        self.blob = torch.empty(off, dtype=torch.uint8, device=device, pin_memory=pinned)
        self.views = {}
        for (name, shape, dtype), o in zip(specs, self.offsets):
            n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            self.views[name] = self.blob[o:o + n].view(dtype).view(shape)


class GpuStep:
    """Device-resident inputs, outputs and workspaces of one step, and the three
    C-ABI calls that make it up.  The inputs that change every step (logits, Q and
    the fresh K/V rows) share one device buffer, and so do the step's results."""

    def __init__(self, nat, w: synth.Workload, st, logits, att, device, stream):
        import torch
        self.nat, self.w, self.torch = nat, w, torch
        self.dev = device
        self.stream = stream

        def up(a):
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)

        self.up = up
        B, L, N, n = w.batch, w.seq_len, w.n_rows, w.n_unmask
        i32, f32, u8 = torch.int32, torch.float32, torch.uint8
        def tdtype(a):  # bf16 arrays are held as uint16 bit patterns
            return torch.bfloat16 if a.dtype == np.uint16 else torch.from_numpy(a.ravel()[:0]).dtype

        self.in_specs = [("logits", logits.shape, tdtype(logits)), ("q", att.q.shape, tdtype(att.q)),
                         ("k_new", att.k_new.shape, tdtype(att.k_new)),
                         ("v_new", att.v_new.shape, tdtype(att.v_new))]
        self.inputs = Packed(self.in_specs, device)
        for name, a in (("logits", logits), ("q", att.q), ("k_new", att.k_new), ("v_new", att.v_new)):
            self.inputs.views[name].copy_(up(a))
        self.out_specs = [("token", (N,), i32), ("conf", (N,), f32), ("entropy", (N,), f32),
                          ("unmask", (B * n,), i32), ("emax", (B,), f32), ("refresh", (B,), u8),
                          ("idx_next", (B, L), i32), ("count_next", (B,), i32),
                          ("out", att.q.shape, self.inputs.views["q"].dtype)]
        self.results = Packed(self.out_specs, device)
        r = self.results.views
        self.logits = self.inputs.views["logits"]
        self.offsets = up(st.seq_row_offsets)
        self.row_pos = up(st.row_pos)
        self.is_masked = up(st.is_masked)
        self.tokens = up(st.tokens)
        self.decode_step = up(st.decode_step)
        self.step_index = st.step
        self.token, self.conf, self.entropy = r["token"], r["conf"], r["entropy"]
        self.unmask, self.emax, self.refresh = r["unmask"], r["emax"], r["refresh"]
        self.refresh.zero_()
        self.ws_dec = nat.new_workspace(nat.ec_decode_workspace_size(N, B), device)
        self.q, self.k_new, self.v_new = (self.inputs.views[k] for k in ("q", "k_new", "v_new"))
        self.k_cache, self.v_cache = up(att.k_cache), up(att.v_cache)
        self.out = r["out"]
        self.out.zero_()
        self.ws_att = nat.new_workspace(
            nat.ec_attention_workspace_size(B, L, w.r_max, w.n_heads, w.n_kv_heads,
                                           w.head_dim), device)
        # this step's recompute set: built once from the initial state
        self.idx = torch.empty((B, L), dtype=i32, device=device)
        self.count = torch.empty(B, dtype=i32, device=device)
        nat.ec_build_recompute_set(self.is_masked, self.decode_step, self.refresh, st.block_lo,
                                   st.block_hi, w.k, self.idx, self.count)
        self.idx_next, self.count_next = r["idx_next"], r["count_next"]
        self.block = (st.block_lo, st.block_hi)
        self.scale = 1.0 / math.sqrt(w.head_dim)
        torch.cuda.synchronize(device)
        got = self.count.cpu().numpy()
        assert (got == w.r_max).all(), f"recompute set size {got} != {w.r_max}"
        # the three calls of a step, validated and marshalled once
        self.attention = nat.prepare_selective_attention(
            self.q, self.k_new, self.v_new, self.idx, self.count, self.k_cache, self.v_cache,
            self.out, self.scale, self.ws_att, stream=stream)
        self.decode = nat.prepare_decode_step(
            self.logits, self.offsets, self.row_pos, w.seq_len, w.n_unmask, w.tau,
            self.step_index, self.token, self.conf, self.entropy, self.unmask, self.emax,
            self.refresh, self.is_masked, self.tokens, self.decode_step, self.ws_dec,
            stream=stream)
        self.recompute = nat.prepare_build_recompute_set(
            self.is_masked, self.decode_step, self.refresh, self.block[0], self.block[1], w.k,
            self.idx_next, self.count_next, stream=stream)

    def run(self):
        self.attention()
        self.decode()
        self.recompute()


def kernels_per_step(nat, w: synth.Workload):
    """Launches of our kernels per step, as the library reports them (the bf16
    attention call is one kernel; float32 runs a write-back and the CUDA-core
    kernel)."""
    import torch
    dt = torch.bfloat16 if w.attn_dtype == synth.BF16 else torch.float32
    n_att = nat.ec_attention_kernel_count(dt, w.batch, w.seq_len, w.r_max, w.n_heads,
                                          w.n_kv_heads, w.head_dim)
    return {"attention": n_att, "decode": 2 if w.n_rows > 0 else 1, "recompute": 1}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("nccl" if _cuda_ok() else "gloo")
    return rank, world, local


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int) -> float:
    """Max over ranks (CPU tensor through the process group)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    return per_rank_units * world / max_seconds


def run_ours(args, workload=None):
    import torch
    rank, world, local = dist_setup(args)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from entropy_gated_kv_decode_b300 import _native as nat
    nat.lib()  # fails loudly when libec.so is missing: there is no other path
    w = synth.WORKLOADS[workload or args.workload]
    geo = workload_geometry(w)
    st, logits, att = host_inputs(w, args.seed)
    stream = torch.cuda.Stream(device)
    torch.cuda.set_stream(stream)
    step = GpuStep(nat, w, st, logits, att, device, stream)
    flush = L2Flush(device)
    K, W = args.steps, args.warmup

    for _ in range(W):
        flush()
        step.run()
    torch.cuda.synchronize(device)
    # Four CUDA graphs, each one call (or the whole step) between its own pair of
    # timing events: host launch cost stays out of the device time, and within
    # the step graph the calls chain as they do in use (each kernel's set-up
    # overlaps its predecessor's tail).
    parts = {"step": step.run, "attention": step.attention, "decode_gate": step.decode,
             "recompute_set": step.recompute}
    ev = {k: (torch.cuda.Event(enable_timing=True, external=True),
              torch.cuda.Event(enable_timing=True, external=True)) for k in parts}
    graphs = {}
    mode = "cuda-graph replay per call"

    def record(name):
        ev[name][0].record()
        parts[name]()
        ev[name][1].record()

    if args.eager:
        mode = "eager launches"
    else:
        try:
            for name in parts:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    record(name)
                graphs[name] = g
            for g in graphs.values():
                g.replay()
            torch.cuda.synchronize(device)
        except Exception as exc:  # capture not possible: time eager launches instead
            graphs = {}
            mode = f"eager launches (graph capture failed: {type(exc).__name__})"

    def replay(name):
        graphs[name].replay() if graphs else record(name)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(device)
    t_wall = time.perf_counter()
    t = {name: 0.0 for name in parts}
    for _ in range(K):
        for name in parts:
            flush()
            replay(name)
        ev["recompute_set"][1].synchronize()
        for name in parts:
            t[name] += ev[name][0].elapsed_time(ev[name][1]) / 1e3
    torch.cuda.synchronize(device)
    barrier(world)
    wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    t_max = {name: reduce_max(v, world) for name, v in t.items()}
    status = nat.ec_read_device_status(step.ws_dec) | nat.ec_read_device_status(step.ws_att)

    e2e = run_e2e(step, geo, w, logits, att, max(100, args.e2e_steps),
                  max(20, args.e2e_warmup), world)

    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tc = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    us = lambda x: x / K * 1e6  # noqa: E731
    t_att, t_dec = t_max["attention"], t_max["decode_gate"]
    att_tflops = geo["attn_flops"] * K / t_att / 1e12
    att_gbs = geo["attn_bytes"] * K / t_att / 1e9
    att_ai = geo["attn_flops"] / geo["attn_bytes"]
    att_roof = min(tc, att_ai * hbm / 1e3)
    dec_gbs = geo["logits_bytes"] * K / t_dec / 1e9
    n_launch = kernels_per_step(nat, w)
    out_parts = {
        "step": {"us": us(t_max["step"]),
                 "logits_gbs": geo["logits_bytes"] * K / t_max["step"] / 1e9,
                 "launches": sum(n_launch.values())},
        "attention": {"us": us(t_att), "tflops": att_tflops, "frac_tensor_peak": att_tflops / tc,
                      "gbs": att_gbs, "frac_hbm": att_gbs / hbm,
                      "frac_attainable": att_tflops / att_roof, "intensity_flop_per_byte": att_ai,
                      "launches": n_launch["attention"]},
        "decode_gate": {"us": us(t_dec), "gbs": dec_gbs, "frac_hbm": dec_gbs / hbm,
                        "launches": n_launch["decode"]},
        "recompute_set": {"us": us(t_max["recompute_set"]), "launches": 1},
    }
    dominant = "attention" if t_att > t_dec else "decode_gate"
    if dominant == "attention":
        bound = "tensor" if att_ai > tc * 1e3 / hbm else "hbm"
        if bound == "hbm":
            roof = {"bound": "hbm", "achieved": att_gbs, "peak": hbm, "unit": "GB/s",
                    "frac": att_gbs / hbm}
        else:
            roof = {"bound": "tensor", "achieved": att_tflops, "peak": tc, "unit": "TFLOP/s",
                    "frac": att_tflops / tc}
        roof["kernel"] = "ec_selective_attention"
        roof["traffic"] = measured_traffic(w.name, "attention")
    else:
        roof = {"bound": "hbm", "achieved": dec_gbs, "peak": hbm, "unit": "GB/s",
                "frac": dec_gbs / hbm, "kernel": "decode_gate_kernel",
                "traffic": measured_traffic(w.name, "decode")}
    roof["peak_source"] = ("measured burst (MEASURED_PEAKS.json)" if peak_kind == "measured"
                           else "fallback")

    if w.logits_dtype == synth.BF16 and not args.no_lmhead:
        out_parts["lmhead_gate"] = lmhead_part(nat, w, st, device, stream, flush, min(K, 50), tc,
                                               hbm, args.seed)

    if w.attn_dtype == synth.BF16 and not args.no_cover:
        out_parts["cover_attention"] = cover_part(nat, step, st, w, flush, min(K, 200), hbm, tc,
                                                  args.seed)
    if w.attn_dtype == synth.BF16 and args.cover_score:
        out_parts["cover_seed_score"] = cover_score_part(nat, step, st, w, flush, min(K, 200),
                                                         args.seed)
    if w.attn_dtype == synth.BF16 and not args.no_simsd:
        out_parts["simsd_attention"] = simsd_part(nat, device, stream, flush, min(K, 200), tc, hbm,
                                                  args.seed)

    cpu = None
    if rank == 0 and world == 1:
        cpu = cpu_baseline(w, st, logits, att, args.cpu_seconds, geo)

    value = aggregate(geo["logits_bytes"] * K, world, t_dec) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": t_max["step"] / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.attn_dtype == synth.BF16 else "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seq_len": w.seq_len, "vocab": w.vocab,
                   "n_rows": w.n_rows, "recompute_rows": w.r_max, "n_heads": w.n_heads,
                   "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "n_unmask": w.n_unmask,
                   "k": w.k, "tau": w.tau, "accumulate": "f32",
                   "l2": "flushed before every timed replay (256 MiB write + 256 MiB read, untimed)",
                   "launch": mode, "parallelism": f"replicas x{world}"},
        "value_note": "decode-and-gate call: logits bytes / its own device time; "
                      "ms_per_step is the whole step (attention, decode, recompute set)",
        "parts": out_parts,
        "roofline": roof, "clocks": clocks, "e2e": e2e,
        "gpu_launches": (sum(n_launch.values()) * 2) * K,
        "cpu_baseline": cpu, "device_status": status, "wall_s_timed_region": wall,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


LMHEAD_HIDDEN = 4096


def lmhead_part(nat, w: synth.Workload, st, device, stream, flush, K, tc_peak, hbm_peak, seed):
    """The LM-head fused decode-and-gate call on this workload's rows (hidden size
    4096, Gaussian bf16 inputs), against the unfused pair it replaces: a cuBLAS
    GEMM writing bf16 logits, then the decode-and-gate call reading them."""
    import torch
    N, V, Hd, B = w.n_rows, w.vocab, LMHEAD_HIDDEN, w.batch
    x, wl = synth.make_lmhead(np.random.default_rng(seed + 101), N, V, Hd, exact=False)
    as_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)  # noqa: E731
    xd, wd = as_bf16(x), as_bf16(wl)
    del x, wl
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
    off, pos = up(st.seq_row_offsets), up(st.row_pos)
    state = [up(st.is_masked), up(st.tokens), up(st.decode_step)]
    outs = [torch.empty(N, dtype=torch.int32, device=device), torch.empty(N, device=device),
            torch.empty(N, device=device),
            torch.empty(B * w.n_unmask, dtype=torch.int32, device=device),
            torch.empty(B, device=device), torch.empty(B, dtype=torch.uint8, device=device)]
    ws = nat.new_workspace(nat.ec_lmhead_workspace_size(N, V, B), device)
    fused = nat.prepare_lmhead_decode_step(xd, wd, off, pos, w.seq_len, w.n_unmask, w.tau, st.step,
                                           *outs, *state, ws, stream=stream)
    logits = torch.empty((N, V), dtype=torch.bfloat16, device=device)
    ws_dec = nat.new_workspace(nat.ec_decode_workspace_size(N, B), device)
    decode = nat.prepare_decode_step(logits, off, pos, w.seq_len, w.n_unmask, w.tau, st.step,
                                     *outs, *state, ws_dec, stream=stream)

    def unfused_gemm():
        torch.matmul(xd, wd.t(), out=logits)

    unfused_gemm()  # cuBLAS creates its handle and workspace outside the graph capture
    torch.cuda.synchronize(device)

    def timed(fns, reps):
        ev = [(torch.cuda.Event(enable_timing=True, external=True),
               torch.cuda.Event(enable_timing=True, external=True)) for _ in fns]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for f, (e0, e1) in zip(fns, ev):
                e0.record()
                f()
                e1.record()
        for _ in range(3):
            flush()
            g.replay()
        tot = [0.0] * len(fns)
        for _ in range(reps):
            flush()
            g.replay()
            ev[-1][1].synchronize()
            for i, (e0, e1) in enumerate(ev):
                tot[i] += e0.elapsed_time(e1) / 1e3
        return [t / reps * 1e6 for t in tot]

    (t_fused,) = timed([fused], K)
    t_gemm, t_dec = timed([unfused_gemm, decode], K)
    status = nat.ec_read_device_status(ws) | nat.ec_read_device_status(ws_dec)
    flops = 2.0 * N * V * Hd
    w_bytes = V * Hd * 2 + N * Hd * 2
    tflops = flops / t_fused / 1e6
    del xd, wd, logits
    return {"us": t_fused, "hidden": Hd, "tflops": tflops, "frac_tensor_peak": tflops / tc_peak,
            "weight_gbs": w_bytes / t_fused / 1e3, "frac_hbm": w_bytes / t_fused / 1e3 / hbm_peak,
            "logits_bytes_not_moved": 2 * N * V * 2,
            "unfused_us": {"cublas_gemm": t_gemm, "decode_gate": t_dec, "total": t_gemm + t_dec},
            "speedup_vs_unfused": (t_gemm + t_dec) / t_fused, "launches": 1,
            "device_status": status, "inputs": "Gaussian bf16 (hidden N(0,1), W_lm N(0, 4/hidden))"}


def simsd_part(nat, device, stream, flush, K, tc_peak, hbm_peak, seed):
    """The attention call under SimSD's temporal causal mask on its verification
    workload (32 sequences, 1024-token prompt, data and mask sections of 8), and
    the unmasked call on the same inputs for the cost of the mask."""
    import torch
    w = synth.SIMSD
    r = 2 * w.block
    rng = np.random.default_rng(seed + 202)
    section, tau, idx, cnt = synth.make_simsd_layout(rng, w.batch, w.prompt_len, w.block)
    a = synth.make_attention(rng, w, r)
    up = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(device)  # noqa: E731
    as_bf16 = lambda x: up(x.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    q, kn, vn, kc, vc = (as_bf16(x) for x in (a.q, a.k_new, a.v_new, a.k_cache, a.v_cache))
    out = torch.empty_like(q)
    ws = nat.new_workspace(nat.ec_attention_workspace_size(w.batch, w.seq_len, r, w.n_heads,
                                                           w.n_kv_heads, w.head_dim), device)
    scale = 1.0 / math.sqrt(w.head_dim)
    # the prepared calls hold raw pointers: every tensor they use stays referenced here
    idx_d, cnt_d, sec_d, tau_d = up(idx), up(cnt), up(section), up(tau)
    masked = nat.prepare_selective_attention_simsd(q, kn, vn, idx_d, cnt_d, sec_d, tau_d, kc, vc,
                                                   out, scale, ws, stream=stream)
    plain = nat.prepare_selective_attention(q, kn, vn, idx_d, cnt_d, kc, vc, out, scale, ws,
                                            stream=stream)

    def timed(fn):
        e0 = torch.cuda.Event(enable_timing=True, external=True)
        e1 = torch.cuda.Event(enable_timing=True, external=True)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            e0.record()
            fn()
            e1.record()
        for _ in range(3):
            flush()
            g.replay()
        tot = 0.0
        for _ in range(K):
            flush()
            g.replay()
            e1.synchronize()
            tot += e0.elapsed_time(e1) / 1e3
        return tot / K * 1e6

    t_m = timed(masked)
    t_p = timed(plain)
    status = nat.ec_read_device_status(ws)
    B, L, H, Hkv, d = w.batch, w.seq_len, w.n_heads, w.n_kv_heads, w.head_dim
    nbytes = (2 * B * L * Hkv * d + 2 * B * r * H * d + 4 * B * r * Hkv * d) * 2
    gbs = nbytes / t_m / 1e3
    return {"us": t_m, "gbs": gbs, "frac_hbm": gbs / hbm_peak, "algorithmic_bytes": nbytes,
            "tflops": 4.0 * B * r * L * H * d / t_m / 1e6, "unmasked_us": t_p,
            "launches": 1, "device_status": status,
            "config": {"batch": B, "prompt": w.prompt_len, "sections": w.block, "seq_len": L,
                       "query_rows": r, "n_heads": H, "n_kv_heads": Hkv, "head_dim": d}}


def cover_part(nat, step, st, w, flush, K, hbm_peak, tc_peak, seed, n_seeds=8):
    """The attention call with COVER's dual view on this workload's recompute set,
    ``n_seeds`` seeds per sequence among its decoded rows, and the plain call on
    the same inputs for the cost of the override."""
    import torch
    torch.cuda.synchronize()
    idx_h, cnt_h = step.idx.cpu().numpy(), step.count.cpu().numpy()
    r = w.r_max
    seeds = synth.cover_seeds(np.random.default_rng(seed + 303), st.is_masked, idx_h, cnt_h, r,
                              n_seeds)
    dev = step.dev
    seed_d = torch.from_numpy(seeds).to(dev)
    kc, vc = step.k_cache.clone(), step.v_cache.clone()
    out = torch.empty_like(step.out)
    ws = nat.new_workspace(nat.ec_attention_workspace_size(w.batch, w.seq_len, r, w.n_heads,
                                                           w.n_kv_heads, w.head_dim), dev)
    scale = 1.0 / math.sqrt(w.head_dim)
    cover = nat.prepare_selective_attention_cover(step.q, step.k_new, step.v_new, step.idx,
                                                  step.count, seed_d, kc, vc, out, scale, ws,
                                                  stream=step.stream)
    plain = nat.prepare_selective_attention(step.q, step.k_new, step.v_new, step.idx, step.count,
                                            kc, vc, out, scale, ws, stream=step.stream)

    def timed(fn):
        e0 = torch.cuda.Event(enable_timing=True, external=True)
        e1 = torch.cuda.Event(enable_timing=True, external=True)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=step.stream):
            e0.record()
            fn()
            e1.record()
        for _ in range(3):
            flush()
            g.replay()
        tot = 0.0
        for _ in range(K):
            flush()
            g.replay()
            e1.synchronize()
            tot += e0.elapsed_time(e1) / 1e3
        return tot / K * 1e6

    t_c = timed(cover)
    t_p = timed(plain)
    geo = workload_geometry(w)
    tflops = geo["attn_flops"] / t_c / 1e6
    return {"us": t_c, "tflops": tflops, "frac_tensor_peak": tflops / tc_peak,
            "gbs": geo["attn_bytes"] / t_c / 1e3, "frac_hbm": geo["attn_bytes"] / t_c / 1e3 / hbm_peak,
            "plain_us": t_p, "seeds_per_sequence": n_seeds, "launches": 1,
            "device_status": nat.ec_read_device_status(ws)}


# float32 FMA peak of the SIMT pipes: 148 SMs x 128 lanes x 2 flops x 2.032 GHz
FP32_SIMT_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def cover_score_part(nat, step, st, w, flush, K, seed, n_drafted=4, n_seed=8):
    """COVER's seed score on this workload's recompute set after the step's
    attention: ``n_drafted`` masked rows per sequence drafted at this step, the
    rest still masked, the decoded rows candidates.  float32 SIMT work: one
    q . k per (active row, head, key) and per (candidate, head, masked row)."""
    import torch
    torch.cuda.synchronize()
    idx_h, cnt_h = step.idx.cpu().numpy(), step.count.cpu().numpy()
    r = w.r_max
    role, drafted, u = synth.cover_score_inputs(np.random.default_rng(seed + 404), st.is_masked,
                                                idx_h, cnt_h, r, n_drafted)
    dev = step.dev
    role_d, drafted_d, u_d = (torch.from_numpy(a).to(dev) for a in (role, drafted, u))
    outs = [torch.empty((w.batch, r), dtype=torch.float32, device=dev) for _ in range(3)]
    seeds = torch.empty((w.batch, n_seed), dtype=torch.int32, device=dev)
    ws = nat.new_workspace(nat.ec_cover_score_workspace_size(w.batch, w.seq_len, r, w.n_heads), dev)
    call = nat.prepare_cover_seed_score(step.q, step.k_cache, step.idx, step.count, role_d,
                                        drafted_d, u_d, 1.0 / math.sqrt(w.head_dim), n_seed,
                                        outs[0], outs[1], outs[2], seeds, ws, stream=step.stream)
    e0 = torch.cuda.Event(enable_timing=True, external=True)
    e1 = torch.cuda.Event(enable_timing=True, external=True)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=step.stream):
        e0.record()
        call()
        e1.record()
    for _ in range(3):
        flush()
        g.replay()
    tot = 0.0
    for _ in range(K):
        flush()
        g.replay()
        e1.synchronize()
        tot += e0.elapsed_time(e1) / 1e3
    us = tot / K * 1e6
    flops = 0.0
    for b in range(w.batch):
        rows = role[b, :int(cnt_h[b])]
        active, cand, masked = (int(np.count_nonzero(rows & 3)), int(np.count_nonzero(rows & 2)),
                                int(np.count_nonzero(rows & 1)))
        flops += 2.0 * w.head_dim * w.n_heads * (active * w.seq_len + cand * masked)
    tflops = flops / us / 1e6
    return {"us": us, "tflops_fp32": tflops, "frac_fp32_simt_peak": tflops / FP32_SIMT_TFLOPS,
            "peak_source": "derived: 148 SMs x 128 FP32 lanes x 2 x 2.032 GHz",
            "drafted_per_sequence": n_drafted, "n_seed": n_seed,
            "launches": nat.ec_cover_score_kernel_count(w.batch, r, n_seed),
            "device_status": nat.ec_read_device_status(ws)}


def run_e2e(step: GpuStep, geo, w, logits, att, K, W, world):
    """Same metric through the public calls, starting from pinned host buffers:
    every step copies its inputs host->device and its results device->host.
    W untimed steps first, then K steps each between its own events (L2 flushed
    before each, outside the events); the value uses the median step time."""
    import torch
    dev = step.dev

    def host(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a))

    # the step's inputs in one pinned buffer with the device buffer's layout, and
    # one pinned buffer for its results: one copy each way per step
    h_in = Packed(step.in_specs, "cpu", pinned=True)
    for name, a in (("logits", logits), ("q", att.q), ("k_new", att.k_new), ("v_new", att.v_new)):
        h_in.views[name].copy_(host(a))
    h_out = Packed(step.out_specs, "cpu", pinned=True)
    bi, bo = h_in.nbytes, h_out.nbytes
    flush = L2Flush(dev)

    def one():
        step.inputs.blob.copy_(h_in.blob, non_blocking=True)
        step.run()
        h_out.blob.copy_(step.results.blob, non_blocking=True)

    for _ in range(W):
        flush()
        one()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    barrier(world)
    for i in range(K):
        flush()
        ev[i][0].record()
        one()
        ev[i][1].record()
    torch.cuda.synchronize(dev)
    barrier(world)
    per = sorted(a.elapsed_time(b) / 1e3 for a, b in ev)
    med = reduce_max(per[len(per) // 2], world)
    mean = reduce_max(sum(per) / len(per), world)
    return {"value": aggregate(geo["logits_bytes"], world, med) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": K, "warmup": W,
            "ms_per_step": med * 1e3, "ms_per_step_median": med * 1e3,
            "ms_per_step_mean": mean * 1e3,
            "note": "whole step (3 calls) plus one pinned copy each way; value from the median"}


# ---------------------------------------------------------------------------
# the float64 CPU oracle as the reported baseline / reference arm


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_step_seconds(orc, w, st, logits, att, budget_s, rng, threads=1):
    """Seconds the float64 oracle takes for one full step on `threads` host
    threads, measured on a bounded sample: entropy rows and attention (row, head)
    outputs are each timed on as many items as half the budget allows (at least
    four per thread) and scaled to the full count; the unmask/gate, index-set
    and write-back stages run in full.
    Returns (seconds per full step, description of the sample)."""
    orc.set_threads(threads)
    N = w.n_rows
    t0 = time.perf_counter()
    orc.row_stats(logits[:1])
    per_row = max(time.perf_counter() - t0, 1e-6) / threads
    n_rows = int(min(N, max(4 * threads, 0.5 * budget_s / per_row)))
    t0 = time.perf_counter()
    h, c, t = orc.row_stats(logits[:n_rows])
    t_rows = (time.perf_counter() - t0) / n_rows * N
    h, c, t = np.resize(h, N), np.resize(c, N), np.resize(t, N)
    t0 = time.perf_counter()
    g = orc.unmask_gate(c, h, t, st.seq_row_offsets, st.row_pos, w.seq_len, w.n_unmask, w.tau,
                        st.step, st.is_masked, st.tokens, st.decode_step)
    orc.recompute_set(g["is_masked"], g["decode_step"], g["refresh"], st.block_lo, st.block_hi,
                      w.k)
    idx, cnt = orc.recompute_set(st.is_masked, st.decode_step, np.zeros(w.batch, np.uint8),
                                 st.block_lo, st.block_hi, w.k)
    kc, vc = orc.scatter_kv(att.k_new, att.v_new, idx, cnt, att.k_cache, att.v_cache)
    t_rest = time.perf_counter() - t0
    scale = 1.0 / math.sqrt(w.head_dim)
    total = int(cnt.sum()) * w.n_heads

    def triples(ids):
        out = []
        for i in ids:
            hh = int(i) % w.n_heads
            rr = int(i) // w.n_heads
            b = 0
            while rr >= cnt[b]:
                rr -= cnt[b]
                b += 1
            out.append((b, rr, hh))
        return np.array(out, np.int32)

    t0 = time.perf_counter()
    orc.attention(att.q, kc, vc, cnt, scale, samples=triples(rng.choice(total, size=1)))
    per_out = max(time.perf_counter() - t0, 1e-6) / threads
    n_out = int(min(total, max(4 * threads, 0.5 * budget_s / per_out)))
    pick = triples(rng.choice(total, size=n_out, replace=False))
    t0 = time.perf_counter()
    orc.attention(att.q, kc, vc, cnt, scale, samples=pick)
    t_att = (time.perf_counter() - t0) / n_out * total
    orc.set_threads(1)
    sample = (f"entropy on {n_rows}/{N} logits rows, attention on {n_out}/{total} (row, head) "
              f"outputs, each scaled to the full step; unmask, gate, index set, write-back in full")
    return t_rows + t_rest + t_att, sample


def cpu_baseline(w, st, logits, att, budget_s, geo):
    """The oracle timed on one host core and on every core this process may use."""
    import oracle as orc
    orc.build()
    cores = orc.usable_cores()
    one, sample1 = oracle_step_seconds(orc, w, st, logits, att, budget_s, np.random.default_rng(1), 1)
    every, sample_n = oracle_step_seconds(orc, w, st, logits, att, budget_s,
                                          np.random.default_rng(2), cores)
    return {"value": geo["logits_bytes"] / every / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle", "sample": sample_n, "seconds_per_step": every,
            "single_core": {"value": geo["logits_bytes"] / one / 1e9, "unit": "GB/s", "cores": 1,
                            "sample": sample1, "seconds_per_step": one},
            "cpu_model": cpu_model(),
            "note": "OpenMP over independent rows and (row, head) outputs; value = all cores"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = synth.WORKLOADS[DEFAULT_WORKLOAD if args.workload == "all" else args.workload]
    if w.name == "trajectory":
        w = synth.WORKLOADS[DEFAULT_WORKLOAD]
    geo = workload_geometry(w)
    st, logits, att = host_inputs(w, args.seed)
    import oracle as orc
    orc.build()
    cores = orc.usable_cores()
    # the whole run (warm-up + K sampled steps) takes about --cpu-seconds x 12
    budget = max(0.005, 12 * args.cpu_seconds / max(1, args.steps + args.warmup))
    rng = np.random.default_rng(1)
    for _ in range(args.warmup):
        oracle_step_seconds(orc, w, st, logits, att, budget, rng, cores)
    times, sample = [], ""
    for _ in range(args.steps):
        s, sample = oracle_step_seconds(orc, w, st, logits, att, budget, rng, cores)
        times.append(s)
    t = sum(times)
    value = geo["logits_bytes"] * len(times) / t / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t / len(times) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seq_len": w.seq_len, "vocab": w.vocab,
                   "n_rows": w.n_rows, "recompute_rows": w.r_max, "n_heads": w.n_heads,
                   "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the multi-step trajectory workload


def trajectory_bytes(w):
    rows = synth.trajectory_rows_per_step(w)
    return sum(rows) * w.vocab * 2


def time_projection(nat, tr, rows, reps=20):
    """Mean device time (s) of one full-shape Q/K/V projection launch, on the
    trajectory's stream with its own buffers (the launch the forward makes)."""
    import torch
    calls = tr.forward_full if rows == tr.w.seq_len else tr.forward_sel
    proj = calls[1]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(tr.stream):
        proj()
        e0.record()
        for _ in range(reps):
            proj()
        e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps


def time_forward(tr, full: bool, reps=10):
    """Mean device time (s) of one forward variant (graph replay), over reps
    replays with the trajectory's buffers."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(tr.stream):
        tr._forward(full)
        e0.record()
        for _ in range(reps):
            tr._forward(full)
        e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps


def trajectory_cpu_baseline(w, seed, budget_s, total_bytes):
    """The oracle's decision path (row statistics, unmasking, gate, index sets;
    no layers) on one core and on all cores, over the first steps that fit the
    budget, scaled to the whole trajectory by logits rows."""
    import oracle as orc
    import oracle.trajectory as otr
    orc.build()
    rows = synth.trajectory_rows_per_step(w)
    cores = orc.usable_cores()
    out = {}
    for threads in (1, cores):
        orc.set_threads(threads)
        n = 1
        while True:
            t0 = time.perf_counter()
            otr.run(w, seed, n_steps=n)
            dt = time.perf_counter() - t0
            if dt > 0.25 * budget_s or n >= w.n_steps:
                break
            n = min(w.n_steps, n * 2)
        secs = dt * sum(rows) / max(1, sum(rows[:n]))
        out[threads] = (secs, f"decision path of the first {n}/{w.n_steps} steps scaled by "
                              f"logits rows; the layers' forward is not timed")
    orc.set_threads(1)
    secs, sample = out[cores]
    one, sample1 = out[1]
    return {"value": total_bytes / secs / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": sample, "seconds_per_trajectory": secs,
            "single_core": {"value": total_bytes / one / 1e9, "unit": "GB/s", "cores": 1,
                            "sample": sample1, "seconds_per_trajectory": one},
            "cpu_model": cpu_model()}


def run_trajectory(args):
    import torch
    rank, world, local = dist_setup(args)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from entropy_gated_kv_decode_b300 import _native as nat
    from entropy_gated_kv_decode_b300.trajectory import Trajectory
    nat.lib()
    w = synth.WORKLOADS["trajectory"]
    stream = torch.cuda.Stream(device)
    torch.cuda.set_stream(stream)
    tr = Trajectory(w, seed=args.seed, device=device, stream=stream)
    tr.warm_up()
    K, W = max(1, args.steps), max(3, args.warmup)
    for _ in range(W):
        tr.run()
    sampler = ClockSampler(None)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(device)
    recs_all, walls = [], []
    for _ in range(K):
        t0 = time.perf_counter()
        recs_all.append(tr.run())
        walls.append(time.perf_counter() - t0)
    torch.cuda.synchronize(device)
    barrier(world)
    clocks = sampler.stop()
    recs = recs_all[-1]
    fwd = sum(r.forward_ms for rr in recs_all for r in rr) / 1e3
    dec = sum(r.decode_ms for rr in recs_all for r in rr) / 1e3
    device_s = fwd + dec
    wall = sum(walls)
    t_max = reduce_max(wall, world)
    n_steps = w.n_steps * K
    full = [r for r in recs if r.full]
    sel = [r for r in recs if not r.full]
    t_proj_full = time_projection(nat, tr, w.seq_len)
    t_proj_sel = time_projection(nat, tr, tr.r_sel)
    t_fwd_full = time_forward(tr, True)
    t_fwd_sel = time_forward(tr, False)
    # end to end: each step's logits copied in from pinned host memory inside the
    # step, the one-byte flag (and the next row count) read back every step
    tr.use_host_logits(True)
    tr.run()
    torch.cuda.synchronize(device)
    e2e_walls = []
    for _ in range(max(2, min(K, 5))):
        t0 = time.perf_counter()
        tr.run()
        tok = tr.tokens.cpu()
        e2e_walls.append(time.perf_counter() - t0)
    tr.use_host_logits(False)
    del tok
    e2e_wall = reduce_max(sorted(e2e_walls)[len(e2e_walls) // 2], world)
    peaks, peak_kind = load_peaks()
    tc = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hid = w.n_heads * w.head_dim
    flops_full = 2.0 * w.seq_len * hid * 3 * hid
    proj_tflops = flops_full / t_proj_full / 1e12
    wbytes = 3 * hid * hid * 2
    tbytes = trajectory_bytes(w)
    value = aggregate(tbytes * K, world, t_max) / 1e9
    cpu = trajectory_cpu_baseline(w, args.seed, args.cpu_seconds, tbytes) \
        if rank == 0 and world == 1 else None
    # the same trajectory under the sliding-window and multi-block decoding policies
    policies = {}
    for pol in (("sliding", 64), ("multiblock", 2)):
        tp = Trajectory(w, seed=args.seed, device=device, stream=stream, policy=pol)
        tp.warm_up()
        tp.run()
        torch.cuda.synchronize(device)
        pw = []
        for _ in range(max(1, min(K, 3))):
            t0 = time.perf_counter()
            pr = tp.run()
            pw.append(time.perf_counter() - t0)
        policies[f"{pol[0]}_{pol[1]}"] = {
            "denoising_steps_per_s": w.n_steps / (sum(pw) / len(pw)),
            "refresh_fraction": sum(r.refresh for r in pr) / len(pr),
            "mean_rows": float(np.mean([r.rows for r in pr])),
            "decode_and_sets_ms": float(np.mean([r.decode_ms for r in pr]))}
        del tp
    # the same trajectory with pre-norm layers (norms, rotary embedding, output
    # projection, SwiGLU MLP of width 12288): its full forward, and the MLP's two
    # contractions alone (launch indices in the layer's call list: 7 and 8)
    wl = synth.scaled(w, ffn=12288)
    tl = Trajectory(wl, seed=args.seed, device=device, stream=stream)
    tl.warm_up()
    tl.run()
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    lr = tl.run()
    lwall = time.perf_counter() - t0
    t_lfull = time_forward(tl, True, reps=3)

    def time_call(call, reps=10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            call()
            e0.record()
            for _ in range(reps):
                call()
            e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3 / reps

    t_gu = time_call(tl.forward_full[7])
    t_down = time_call(tl.forward_full[8])
    prenorm = {
        "denoising_steps_per_s": wl.n_steps / lwall,
        "refresh_fraction": sum(r.refresh for r in lr) / len(lr),
        "full_forward_ms_replay": t_lfull * 1e3,
        "mlp_gate_up_swiglu_us": t_gu * 1e6,
        "mlp_gate_up_tflops": 2.0 * wl.seq_len * hid * 2 * wl.ffn / t_gu / 1e12,
        "mlp_down_residual_us": t_down * 1e6,
        "mlp_down_tflops": 2.0 * wl.seq_len * wl.ffn * hid / t_down / 1e12,
        "layer": "rms_norm, qkv, rope, attention, o-proj + residual, rms_norm, SwiGLU, down + residual",
        "weights": "drawn on the device (seeded), N(0, 1/fan_in)"}
    del tl
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": t_max / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "trajectory", "seq_len": w.seq_len, "vocab": w.vocab,
                   "denoising_steps": w.n_steps, "layers": w.n_layers, "n_heads": w.n_heads,
                   "head_dim": w.head_dim, "hidden": hid, "n_unmask": w.n_unmask, "k": w.k,
                   "tau": w.tau, "step": "one whole 128-step trajectory",
                   "l2": "inputs (3.2 GB of weights per step) exceed L2",
                   "parallelism": f"replicas x{world}"},
        "value_note": "logits bytes of all 128 denoising steps / wall time of the trajectory",
        "parts": {
            "denoising_steps_per_s": n_steps / wall,
            "refresh_fraction": sum(r.refresh for r in recs) / len(recs),
            "full_forward_steps": len(full), "partial_forward_steps": len(sel),
            "mean_rows": float(np.mean([r.rows for r in recs])),
            "full_forward_ms": float(np.mean([r.forward_ms for r in full])) if full else None,
            "partial_forward_ms": float(np.mean([r.forward_ms for r in sel])) if sel else None,
            "full_forward_ms_replay": t_fwd_full * 1e3,
            "partial_forward_ms_replay": t_fwd_sel * 1e3,
            "partial_forward_rows": tr.r_sel,
            "decode_and_sets_ms": float(np.mean([r.decode_ms for r in recs])),
            "gate_share_of_device_time": dec / device_s,
            "host_overhead_share": max(0.0, 1 - device_s / wall),
            "projection_full_us": t_proj_full * 1e6, "projection_full_tflops": proj_tflops,
            "projection_partial_us": t_proj_sel * 1e6,
            "projection_partial_weight_gbs": wbytes / t_proj_sel / 1e9,
            "policies": policies,
            "prenorm_layers": prenorm,
        },
        "roofline": {"bound": "tensor", "achieved": proj_tflops, "peak": tc, "unit": "TFLOP/s",
                     "frac": proj_tflops / tc, "traffic": None,
                     "kernel": "qkv_gemm_kernel (full-refresh shape 1024 x 12288 x 4096)",
                     "peak_source": f"{peak_kind} sustained (MEASURED_PEAKS.json)"},
        "clocks": clocks,
        "gpu_launches": sum(1 + 2 * w.n_layers + 4 for _ in recs) * K,
        "e2e": {"value": aggregate(tbytes, world, e2e_wall) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": tbytes / w.n_steps,
                "d2h_bytes_per_step": 5 + tr.tokens.numel() * 4 / w.n_steps,
                "ms_per_trajectory": e2e_wall * 1e3,
                "note": "each step's logits copied from pinned host memory inside the step; "
                        "refresh flag and row count read back every step; tokens at the end"},
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_lmhead(args):
    """The LM-head fused decode-and-gate call alone on the batched workload's rows
    (the default line's lmhead_gate part), for profiling that kernel by itself."""
    import torch
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from entropy_gated_kv_decode_b300 import _native as nat
    nat.lib()
    w = synth.WORKLOADS[DEFAULT_WORKLOAD]
    st = synth.make_state(np.random.default_rng(args.seed), w)
    stream = torch.cuda.Stream(device)
    torch.cuda.set_stream(stream)
    peaks, _ = load_peaks()
    part = lmhead_part(nat, w, st, device, stream, L2Flush(device), max(1, args.steps),
                       float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
                       float(peaks["hbm_gbs"]), args.seed)
    print(json.dumps({"workload": "lmhead", "config": {"rows": w.n_rows, "vocab": w.vocab,
                                                        "hidden": LMHEAD_HIDDEN},
                      "lmhead_gate": part}), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "trajectory":
        run_trajectory(args)
    elif args.workload == "lmhead":
        run_lmhead(args)
    elif args.workload == "all":
        for name in ("tiny", "single_seq", "batched", "long_ctx"):
            run_ours(args, name)
        run_trajectory(args)
    else:
        run_ours(args)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
