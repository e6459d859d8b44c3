"""Multi-step denoising trajectory of a masked diffusion model with EntropyCache
on the GPU: the gate decides every step between a full forward and a partial
one.

"EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
Models" — Italian summary, "Algoritmo di Funzionamento" steps 1-3 (decode,
take the maximum entropy E of the new tokens; E > tau: full forward next,
otherwise recompute only the masked tokens and the k most recent ones; repeat),
and the Arabic technical summary, "Algorithm workflow" phases 1-3.

The model is synthetic: ``n_layers`` layers, each a Q/K/V projection of the
recomputed rows followed by selective bidirectional attention over that
layer's KV cache; a layer's attention output rows are the next layer's input
rows, and layer 0 reads token embeddings.  With ``ffn`` > 0 the layers are
pre-norm transformer blocks instead (the layer of the pages' models):
    a = rms_norm(x, g1); [q|k|v] = a W_qkv^T; rope(q, k); o = attention;
    x += o W_o^T; b = rms_norm(x, g2); x += (silu(b W_gate^T) * b W_up^T) W_down^T
(ec_rms_norm, ec_qkv_projection, ec_rope, ec_selective_attention, ec_linear).  The logits of every step are seeded
random numbers (no LM head), so the decision sequence does not depend on the
layers' numerics.

One step t, all on one CUDA stream:
  forward    rows = every position (t = 0, or the previous gate fired) or the
             recompute set built at t-1; a CUDA graph of ec_embed_rows and, per
             layer, ec_qkv_projection + ec_selective_attention (one graph for
             each of the two row counts, captured once);
  decode     ec_build_recompute_set with k = 0 lists the masked positions of the
             active block (the rows of this step's logits), ec_decode_step
             unmasks and gates, ec_build_recompute_set builds the next forward's
             rows for the block active at t+1;
  branch     the one-byte refresh flag is copied to pinned host memory and read
             after the step, which picks the next forward's graph.
Every arithmetic step runs in libec's kernels; this module only allocates,
launches and reads the flag.

Decoding policies (section 5 "Generalità" of the Italian summary: the skipping
rule applies to sliding-window and block decoding).  A step may unmask only
positions of its window [lo, hi), whose masked positions are also the "currently
masked" part of the next recompute set:
  ("block",)          the workload's block schedule, blocks left to right;
  ("sliding", W)      lo = the first still-masked generated position, hi = lo + W;
  ("multiblock", nb)  lo = the start of the block holding that position, nb blocks;
hi clamped to L.  With the last two the window depends on the state: after each
step this module copies is_masked (one byte per position) to the host with the
refresh flag, places the next window there, and builds the next recompute set
before the next forward.  A step's logits are the first c rows of a W-row
(nb-block) draw, c the masked positions in its window.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

from . import _native as nat
from . import synth


@dataclasses.dataclass
class StepRecord:
    step: int
    full: bool          # this step's forward recomputed every position
    rows: int           # rows recomputed by this step's forward
    refresh: int        # the gate's decision at this step (governs step + 1)
    forward_ms: float
    decode_ms: float


def _up(a: np.ndarray, device) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class Trajectory:
    """Device state and launch plan of one synthetic trajectory (batch 1)."""

    def __init__(self, w: synth.Workload, seed: int = 0, device=None, stream=None,
                 use_graphs: bool = True, trace: bool = False, policy=("block",)):
        if w.batch != 1 or w.n_kv_heads != w.n_heads:
            raise ValueError("the trajectory driver runs one sequence of a multi-head model")
        if policy[0] not in ("block", "sliding", "multiblock") or (
                policy[0] != "block" and (len(policy) != 2 or int(policy[1]) < 1)):
            raise ValueError(f"unknown decoding policy {policy}")
        self.policy = policy
        self.windowed = policy[0] != "block"
        self.w, self.seed = w, seed
        self.dev = torch.device(device if device is not None else "cuda")
        self.stream = stream if stream is not None else torch.cuda.Stream(self.dev)
        L, V, H, d = w.seq_len, w.vocab, w.n_heads, w.head_dim
        self.hidden = H * d
        hid = self.hidden
        # rows of every step's logits draw (window policies) and the largest
        # partial recompute set
        self.win_rows = (policy[1] if policy[0] == "sliding" else policy[1] * w.block) \
            if self.windowed else w.block
        self.r_sel = min(self.win_rows + w.k, L)
        i32, u8, bf = torch.int32, torch.uint8, torch.bfloat16
        dev = self.dev
        self.llama = w.ffn > 0
        with torch.cuda.stream(self.stream):
            self.table = _up(synth.trajectory_embedding(seed, V, hid), dev)
            if self.llama:
                self.layers = [self._layer_weights(seed, layer) for layer in range(w.n_layers)]
                self.weights = torch.stack([lw["w_qkv"] for lw in self.layers])
            else:
                self.weights = torch.empty((w.n_layers, 3 * hid, hid), dtype=bf, device=dev)
                for layer in range(w.n_layers):
                    self.weights[layer].copy_(_up(synth.trajectory_weights(seed, layer, hid, hid), dev))
            self.k_cache = torch.zeros((w.n_layers, 1, L, w.n_kv_heads, d), dtype=bf, device=dev)
            self.v_cache = torch.zeros_like(self.k_cache)
            # every step's logits, resident: rows of step t start at row_off[t]
            if self.windowed:
                self.rows_per_step = [self.win_rows] * w.n_steps  # rows drawn per step
            else:
                self.rows_per_step = synth.trajectory_rows_per_step(w)
            self.row_off = np.concatenate([[0], np.cumsum(self.rows_per_step)]).astype(np.int64)
            self.logits = torch.empty((int(self.row_off[-1]), V), dtype=bf, device=dev)
            for t, n in enumerate(self.rows_per_step):
                if n:
                    draw = (synth.trajectory_window_logits(seed, t, n, V) if self.windowed
                            else synth.trajectory_logits(seed, t, n, V))
                    self.logits[self.row_off[t]:self.row_off[t + 1]].copy_(_up(draw, dev))
            st = synth.trajectory_start(seed, w)
            self.start = st
            self.is_masked = _up(st.is_masked, dev)
            self.tokens = _up(st.tokens, dev)
            self.decode_step = _up(st.decode_step, dev)
            # activations: two hidden-state buffers and q / k / v
            self.xa = torch.zeros((1, L, hid), dtype=bf, device=dev)
            self.xb = torch.zeros_like(self.xa)
            if self.llama:
                self.o = torch.zeros_like(self.xa)
                self.m = torch.zeros((1, L, w.ffn), dtype=bf, device=dev)
            self.q = torch.zeros_like(self.xa)
            self.k = torch.zeros_like(self.xa)
            self.v = torch.zeros_like(self.xa)
            # row sets
            self.idx_full = torch.arange(L, dtype=i32, device=dev).reshape(1, L)
            self.count_full = torch.full((1,), L, dtype=i32, device=dev)
            self.idx_sel = torch.full((1, L), -1, dtype=i32, device=dev)
            self.count_sel = torch.zeros(1, dtype=i32, device=dev)
            self.idx_rows = torch.full((1, L), -1, dtype=i32, device=dev)
            self.count_rows = torch.zeros(1, dtype=i32, device=dev)
            self.zero_flag = torch.zeros(1, dtype=u8, device=dev)
            # decode outputs
            nb = self.win_rows
            if self.windowed:  # offsets [0, c] for every possible row count c
                self.offsets = _up(np.array([[0, c] for c in range(nb + 1)], np.int32), dev)
            else:
                self.offsets = _up(np.array([[0, n] for n in self.rows_per_step], np.int32), dev)
            self.mask_host = torch.zeros((1, L), dtype=u8).pin_memory()
            self.token = torch.zeros(nb, dtype=i32, device=dev)
            self.conf = torch.zeros(nb, dtype=torch.float32, device=dev)
            self.entropy = torch.zeros(nb, dtype=torch.float32, device=dev)
            self.unmask = torch.zeros(w.n_unmask, dtype=i32, device=dev)
            self.emax = torch.zeros(1, dtype=torch.float32, device=dev)
            self.refresh = torch.zeros(1, dtype=u8, device=dev)
            self.refresh_host = torch.zeros(1, dtype=u8).pin_memory()
            self.count_host = torch.zeros(1, dtype=i32).pin_memory()
            # workspaces
            self.ws_dec = nat.new_workspace(nat.ec_decode_workspace_size(nb, 1), dev)
            self.ws_att = nat.new_workspace(max(
                nat.ec_attention_workspace_size(1, L, L, H, w.n_kv_heads, d),
                nat.ec_attention_workspace_size(1, L, self.r_sel, H, w.n_kv_heads, d)), dev)
            self.ws_fwd = nat.new_workspace(256, dev)
        self.scale = 1.0 / math.sqrt(d)
        self.forward_full = self._forward_calls(self.idx_full, self.count_full, L)
        self.forward_sel = self._forward_calls(self.idx_sel, self.count_sel, self.r_sel)
        self.graphs = {}
        self.use_graphs = use_graphs
        self.trace = trace
        self.traces: list[dict] = []
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        self.logits_host = None
        self.copy_logits = False
        self.records: list[StepRecord] = []
        self.t = 0
        self.next_full = True
        self.next_rows = w.seq_len
        self.win = None  # this step's window (window policies)

    def _layer_weights(self, seed: int, layer: int) -> dict:
        """One pre-norm layer's weights on the device: from the shared generator
        for models up to hidden 1024, else drawn on the device (seeded) with the
        same scales, since the host would take minutes for billions of values."""
        w, dev, hid = self.w, self.dev, self.hidden
        if hid <= 1024:
            return {k: _up(v, dev) for k, v in
                    synth.trajectory_layer_weights(seed, layer, hid, w.ffn).items()}
        g = torch.Generator(device=dev)
        g.manual_seed(seed * 1000003 + layer)

        def draw(rows, cols):
            return (torch.randn((rows, cols), generator=g, device=dev) / math.sqrt(cols)).to(torch.bfloat16)

        gains = 1.0 + 0.1 * torch.randn((2, hid), generator=g, device=dev)
        return dict(w_qkv=draw(3 * hid, hid), w_o=draw(hid, hid), w_gu=draw(2 * w.ffn, hid),
                    w_down=draw(hid, w.ffn), g1=gains[0].to(torch.bfloat16).contiguous(),
                    g2=gains[1].to(torch.bfloat16).contiguous())

    # -- launch plan ---------------------------------------------------------

    def _forward_calls(self, idx, count, r):
        """Prepared calls of one forward over `r` row slots (count[0] of them used)."""
        if self.llama:
            return self._llama_calls(idx, count, r)
        w, s = self.w, self.stream
        x = [self.xa[:, :r], self.xb[:, :r]]
        q, k, v = self.q[:, :r], self.k[:, :r], self.v[:, :r]
        H, Hkv, d = w.n_heads, w.n_kv_heads, w.head_dim
        calls = [nat.prepare_embed_rows(self.table, idx, count, self.tokens, self.is_masked,
                                        w.vocab, x[0], self.ws_fwd, stream=s)]
        for layer in range(w.n_layers):
            xin, xout = x[layer % 2], x[(layer + 1) % 2]
            calls.append(nat.prepare_qkv_projection(xin, count, self.weights[layer], q, k, v,
                                                    self.ws_fwd, stream=s))
            calls.append(nat.prepare_selective_attention(
                q.view(1, r, H, d), k.view(1, r, Hkv, d), v.view(1, r, Hkv, d), idx, count,
                self.k_cache[layer], self.v_cache[layer], xout.view(1, r, H, d), self.scale,
                self.ws_att, stream=s))
        return calls

    def _llama_calls(self, idx, count, r):
        """The pre-norm layers: the residual stream stays in xa, xb holds the
        normalised rows."""
        w, s = self.w, self.stream
        H, Hkv, d = w.n_heads, w.n_kv_heads, w.head_dim
        x, a, o, m = self.xa[:, :r], self.xb[:, :r], self.o[:, :r], self.m[:, :r]
        q, k, v = self.q[:, :r], self.k[:, :r], self.v[:, :r]
        ws = self.ws_fwd
        calls = [nat.prepare_embed_rows(self.table, idx, count, self.tokens, self.is_masked,
                                        w.vocab, x, ws, stream=s)]
        for layer, lw in enumerate(self.layers):
            calls += [
                nat.prepare_rms_norm(x, count, lw["g1"], w.norm_eps, a, ws, stream=s),
                nat.prepare_qkv_projection(a, count, lw["w_qkv"], q, k, v, ws, stream=s),
                nat.prepare_rope(q.view(1, r, H, d), k.view(1, r, Hkv, d), idx, count, w.seq_len,
                                 w.rope_theta, ws, stream=s),
                nat.prepare_selective_attention(
                    q.view(1, r, H, d), k.view(1, r, Hkv, d), v.view(1, r, Hkv, d), idx, count,
                    self.k_cache[layer], self.v_cache[layer], o.view(1, r, H, d), self.scale,
                    self.ws_att, stream=s),
                nat.prepare_linear(o, count, lw["w_o"], nat.LINEAR_RESIDUAL, x, x, ws, stream=s),
                nat.prepare_rms_norm(x, count, lw["g2"], w.norm_eps, a, ws, stream=s),
                nat.prepare_linear(a, count, lw["w_gu"], nat.LINEAR_SWIGLU, None, m, ws, stream=s),
                nat.prepare_linear(m, count, lw["w_down"], nat.LINEAR_RESIDUAL, x, x, ws, stream=s),
            ]
        return calls

    def _forward(self, full: bool):
        key = "full" if full else "sel"
        calls = self.forward_full if full else self.forward_sel
        if not self.use_graphs:
            for c in calls:
                c()
            return
        g = self.graphs.get(key)
        if g is None:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for c in calls:
                    c()
            self.graphs[key] = g
        g.replay()

    def use_host_logits(self, on: bool = True):
        """Keep every step's logits in pinned host memory and copy each step's rows
        to the device inside the step, as a caller whose logits arrive from the
        host would (the end-to-end measurement)."""
        if on and self.logits_host is None:
            self.logits_host = torch.empty(self.logits.shape, dtype=self.logits.dtype).pin_memory()
            self.logits_host.copy_(self.logits)
        self.copy_logits = on

    def _window_of(self, mask: np.ndarray) -> tuple[int, int, int]:
        """The window [lo, hi) placed on a host copy of is_masked, and the number of
        masked positions in it."""
        w, pol = self.w, self.policy
        gen = np.flatnonzero(mask[w.prompt_len:])
        first = w.prompt_len + int(gen[0]) if gen.size else w.seq_len
        if pol[0] == "sliding":
            lo = first
        else:
            lo = w.prompt_len + (first - w.prompt_len) // w.block * w.block
        hi = min(lo + self.win_rows, w.seq_len)
        return lo, hi, int(mask[lo:hi].sum())

    def _decode(self, t: int):
        """Unmask and gate with step t's logits, then build the next row set."""
        w = self.w
        if self.windowed:
            lo, hi, n_rows = self.win
        else:
            lo, hi = synth.trajectory_block(w, t)
            n_rows = self.rows_per_step[t]
        if self.copy_logits and n_rows:
            a = int(self.row_off[t])
            self.logits[a:a + n_rows].copy_(self.logits_host[a:a + n_rows], non_blocking=True)
        nat.ec_build_recompute_set(self.is_masked, self.decode_step, self.zero_flag, lo, hi, 0,
                                   self.idx_rows, self.count_rows, stream=self.stream)
        lg = self.logits[self.row_off[t]:self.row_off[t] + n_rows]
        offs = self.offsets[n_rows] if self.windowed else self.offsets[t]
        nat.ec_decode_step(lg, offs, self.idx_rows[0, :n_rows], w.seq_len, w.n_unmask,
                           w.tau, t, self.token[:n_rows], self.conf[:n_rows],
                           self.entropy[:n_rows], self.unmask, self.emax, self.refresh,
                           self.is_masked, self.tokens, self.decode_step, self.ws_dec,
                           stream=self.stream)
        if self.windowed:  # the next window is placed on the host after the step
            self.mask_host.copy_(self.is_masked, non_blocking=True)
        else:
            nlo, nhi = synth.trajectory_block(w, t + 1)
            nat.ec_build_recompute_set(self.is_masked, self.decode_step, self.refresh, nlo, nhi,
                                       w.k, self.idx_sel, self.count_sel, stream=self.stream)
            self.count_host.copy_(self.count_sel, non_blocking=True)
        self.refresh_host.copy_(self.refresh, non_blocking=True)

    def _next_window(self):
        """Window policies, after a step: the next window from the host copy of
        is_masked, and the next recompute set for it (queued before the next
        forward)."""
        lo, hi, c = self._window_of(self.mask_host[0].numpy())
        self.win = (lo, hi, c)
        w = self.w
        with torch.cuda.stream(self.stream):
            nat.ec_build_recompute_set(self.is_masked, self.decode_step, self.refresh, lo, hi, w.k,
                                       self.idx_sel, self.count_sel, stream=self.stream)
            self.count_host.copy_(self.count_sel, non_blocking=True)

    # -- driving -------------------------------------------------------------

    def warm_up(self):
        """Run each forward variant once (eagerly) so graph capture sees warm
        state, then restore the starting state."""
        with torch.cuda.stream(self.stream):
            for c in self.forward_full + self.forward_sel:
                c()
            self.reset()
            if self.use_graphs:
                self._forward(True)
                self._forward(False)
                self.reset()
        torch.cuda.synchronize(self.dev)

    def reset(self):
        """Back to the starting state (caches are rebuilt by step 0's full forward)."""
        st = self.start
        self.is_masked.copy_(_up(st.is_masked, self.dev))
        self.tokens.copy_(_up(st.tokens, self.dev))
        self.decode_step.copy_(_up(st.decode_step, self.dev))
        self.count_sel.zero_()
        self.t = 0
        self.next_full = True
        self.next_rows = self.w.seq_len
        self.records = []
        self.traces = []
        if self.windowed:
            self.win = self._window_of(st.is_masked[0])

    def step(self):
        t = self.t
        ev = self.events
        full, rows = self.next_full, self.next_rows
        with torch.cuda.stream(self.stream):
            ev[0].record()
            self._forward(full)
            ev[1].record()
            self._decode(t)
            ev[2].record()
        ev[2].synchronize()
        refresh = int(self.refresh_host[0])
        self.records.append(StepRecord(t, full, rows, refresh, ev[0].elapsed_time(ev[1]),
                                       ev[1].elapsed_time(ev[2])))
        n = self.win[2] if self.windowed else self.rows_per_step[t]
        if self.windowed:
            self._next_window()
            self.stream.synchronize()  # the next set's size (for the records) has landed
        self.next_full = refresh != 0
        self.next_rows = self.w.seq_len if self.next_full else int(self.count_host[0])
        if self.trace:  # host copies of this step's decisions (outside any timing)
            self.traces.append(dict(
                row_pos=self.idx_rows[0, :n].cpu().numpy(), token=self.token[:n].cpu().numpy(),
                entropy=self.entropy[:n].cpu().numpy(), conf=self.conf[:n].cpu().numpy(),
                unmask_rows=self.unmask.cpu().numpy(), max_entropy=float(self.emax.item()),
                refresh=refresh, idx_next=self.idx_sel[0, :int(self.count_host[0])].cpu().numpy()))
        self.t = t + 1

    def run(self, n_steps: int | None = None):
        """Run the whole trajectory (or its first n_steps) from the starting state."""
        self.reset()
        for _ in range(self.w.n_steps if n_steps is None else n_steps):
            self.step()
        return self.records

    # -- checkpoint / resume ---------------------------------------------------

    _STATE_TENSORS = ("is_masked", "tokens", "decode_step", "k_cache", "v_cache", "idx_sel",
                      "count_sel", "refresh")

    def state_dict(self) -> dict:
        """The state after the last completed step, copied to the host: the decode
        state, every layer's K/V cache, the next forward's row set, the gate flag, the
        step counter and (window policies) the next window.  With the same workload,
        seed and policy, load_state_dict then continues the trajectory exactly as it
        would have gone on."""
        torch.cuda.synchronize(self.dev)
        sd = {name: getattr(self, name).detach().cpu().clone() for name in self._STATE_TENSORS}
        sd.update(t=self.t, next_full=self.next_full, next_rows=self.next_rows, win=self.win,
                  policy=tuple(self.policy), seed=self.seed,
                  workload=dataclasses.asdict(self.w))
        return sd

    def load_state_dict(self, sd: dict):
        """Resume from state_dict(): the next step() is step sd['t']."""
        if (sd["workload"] != dataclasses.asdict(self.w) or sd["seed"] != self.seed
                or tuple(sd["policy"]) != tuple(self.policy)):
            raise ValueError("the checkpoint belongs to another workload, seed or policy")
        with torch.cuda.stream(self.stream):
            for name in self._STATE_TENSORS:
                getattr(self, name).copy_(sd[name].to(self.dev))
        torch.cuda.synchronize(self.dev)
        self.t, self.next_full, self.next_rows = sd["t"], sd["next_full"], sd["next_rows"]
        self.win = sd["win"]
        self.records, self.traces = [], []

    def save(self, path: str):
        torch.save(self.state_dict(), path)

    def load(self, path: str):
        self.load_state_dict(torch.load(path, weights_only=False))
