"""One decode step of a workload, driven through the C ABI.

``DecodeStep`` owns the device-side inputs and outputs of one batch (page
tables, lengths, per-slot sampler state, attention outputs, workspaces) and
runs the hot path: decode_plan once (the batch's attention schedule, shared
by the layers), for every layer kv_append then paged_decode_attn_planned, then
seeded_sample over the logits, then (frame workloads) one frame: a
frame_sample (stop/continue on channel 0, then the codebooks) when the
workload has control logits, else a codebook_frame_sample.  It only orders
calls and allocates buffers with torch; all arithmetic happens in libpkv's
kernels.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from . import _binding as B
from .workloads import Batch, Tensors


class DecodeStep:
    def __init__(self, batch: Batch, tensors: Tensors, device="cuda", stop_tokens=None,
                 audio_lo: int = 0, audio_hi: int = 0, out_fp32: bool = False,
                 with_lse: bool = True, plan_once: bool = True):
        import torch
        cfg = batch.cfg
        self.batch = batch
        self.cfg = cfg
        self.t = tensors
        dev = torch.device(device)
        self.device = dev
        i32 = torch.int32
        self.page_table = torch.as_tensor(batch.page_table, dtype=i32).to(dev)
        self.seq_lens = torch.as_tensor(batch.seq_lens, dtype=i32).to(dev)
        self.active = torch.as_tensor(batch.active, dtype=i32).to(dev)
        self.slots = torch.as_tensor(batch.slots, dtype=i32).to(dev)
        self.seeds = torch.as_tensor(batch.seeds.view(np.int64)).view(torch.uint64).to(dev)
        self.steps = torch.as_tensor(batch.steps, dtype=torch.int64).to(dev)
        self.temperature = torch.as_tensor(batch.temperature).to(dev)
        self.top_k = torch.as_tensor(batch.top_k).to(dev)
        self.top_p = torch.as_tensor(batch.top_p).to(dev)
        self.stop_tokens = (None if not stop_tokens else
                            torch.as_tensor(np.asarray(stop_tokens, np.int32)).to(dev))
        self.audio_lo, self.audio_hi = int(audio_lo), int(audio_hi)
        Bn = batch.B
        L = tensors.layers
        odt = torch.float32 if out_fp32 else torch.bfloat16
        self.out = torch.empty((L, Bn, cfg.num_qo_heads, cfg.head_dim), dtype=odt, device=dev)
        self.lse = (torch.empty((L, Bn, cfg.num_qo_heads), dtype=torch.float32, device=dev)
                    if with_lse else None)
        ws = B.decode_workspace_bytes(Bn, cfg.num_qo_heads, cfg.head_dim, batch.max_pages,
                                      cfg.page_size)
        self.attn_ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.out_tok = torch.empty(Bn, dtype=i32, device=dev)
        self.out_kind = torch.empty(Bn, dtype=i32, device=dev)
        self.samp_ws = None
        if tensors.logits is not None:
            self.samp_ws = torch.empty(B.sample_workspace_bytes(Bn, tensors.logits.shape[1]),
                                       dtype=torch.uint8, device=dev)
        self.frame_ws = None
        if tensors.base is not None:
            n_cb, _, Vf = tensors.base.shape
            if tensors.ctrl is not None:
                # frame rows: channel 0 the control token, then the codes
                nbytes = B.frame_sample_workspace_bytes(n_cb, Bn, Vf, tensors.ctrl.shape[1])
                self.out_codes = torch.empty((Bn, 1 + n_cb), dtype=i32, device=dev)
            else:
                nbytes = B.frame_workspace_bytes(n_cb, Bn, Vf)
                self.out_codes = torch.empty((Bn, n_cb), dtype=i32, device=dev)
            self.frame_ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            self.frame_kind = torch.empty(Bn, dtype=i32, device=dev)
        self.err = torch.zeros(1, dtype=i32, device=dev)
        # plan_once: one decode_plan per step, then the planned attention
        # per layer; else every layer's call plans for itself
        self.plan_once = bool(plan_once)
        self.graph = None
        self._warm = False

    # -- the pieces of the step ------------------------------------------
    def append(self, layer: int, stream=None):
        t = self.t
        B.kv_append(t.cache, layer, t.k[layer], t.v[layer], self.page_table, self.seq_lens,
                    self.active, err_word=self.err, stream=stream)

    def plan(self, stream=None):
        """The batch's attention schedule into the attention workspace."""
        B.decode_plan(self.t.cache, self.cfg.num_qo_heads, self.page_table.shape[1],
                      self.seq_lens, self.active, self.attn_ws, err_word=self.err,
                      stream=stream)

    def attend(self, layer: int, stream=None):
        t = self.t
        B.paged_decode_attn(t.cache, layer, t.q[layer], self.page_table, self.seq_lens,
                            self.active, self.out[layer], self.attn_ws,
                            lse=None if self.lse is None else self.lse[layer],
                            err_word=self.err, stream=stream, planned=self.plan_once)

    def sample(self, advance=True, salt=0, stream=None):
        B.seeded_sample(self.t.logits, self.slots, self.active, self.seeds, self.steps,
                        self.temperature, self.top_k, self.top_p, self.out_tok, self.out_kind,
                        self.samp_ws, salt=salt, advance=advance, stop_tokens=self.stop_tokens,
                        audio_lo=self.audio_lo, audio_hi=self.audio_hi, err_word=self.err,
                        stream=stream)

    def enable_ext(self, min_p=0.05, rep_penalty=1.2, rep_window=-1, hist_cap=256, seed=0):
        """Per-slot settings for sample_ext: the same min_p, penalty and
        window on every slot, and a full history ring of ``hist_cap`` seeded
        random tokens per slot (as after hist_cap generated tokens)."""
        import torch
        dev = self.device
        S = self.seeds.numel()
        V = self.t.logits.shape[1]
        rng = np.random.default_rng(seed)
        self.ext_min_p = torch.full((S,), float(min_p), dtype=torch.float32, device=dev)
        self.ext_pen = torch.full((S,), float(rep_penalty), dtype=torch.float32, device=dev)
        self.ext_window = torch.full((S,), int(rep_window), dtype=torch.int32, device=dev)
        self.ext_history = torch.as_tensor(
            rng.integers(0, V, (S, hist_cap)).astype(np.int32)).to(dev)
        self.ext_hist_len = torch.full((S,), hist_cap, dtype=torch.int32, device=dev)
        Bn = self.batch.B
        self.lp_raw = torch.zeros(Bn, dtype=torch.float32, device=dev)
        self.lp_proc = torch.zeros(Bn, dtype=torch.float32, device=dev)
        self.ext_ws = torch.empty(B.sample_ext_workspace_bytes(Bn, V), dtype=torch.uint8,
                                  device=dev)

    def sample_ext(self, advance=True, salt=0, stream=None):
        """seeded_sample_ext with the settings of enable_ext and both log-probs."""
        B.seeded_sample_ext(self.t.logits, self.slots, self.active, self.seeds, self.steps,
                            self.temperature, self.top_k, self.top_p, self.out_tok,
                            self.out_kind, self.ext_ws, min_p=self.ext_min_p,
                            rep_penalty=self.ext_pen, rep_window=self.ext_window,
                            history=self.ext_history, hist_len=self.ext_hist_len,
                            logprob_raw=self.lp_raw, logprob_proc=self.lp_proc, salt=salt,
                            advance=advance, stop_tokens=self.stop_tokens,
                            audio_lo=self.audio_lo, audio_hi=self.audio_hi, err_word=self.err,
                            stream=stream)

    def frame(self, stream=None):
        t = self.t
        if t.ctrl is not None:
            B.frame_sample(t.ctrl, self.cfg.ctrl_stop, t.base, t.fb, self.slots, self.active,
                           self.seeds, self.steps, self.temperature, self.top_k, self.top_p,
                           self.out_codes, self.frame_kind, self.frame_ws, err_word=self.err,
                           stream=stream)
            return
        B.codebook_frame_sample(t.base, t.fb, self.slots, self.active, self.seeds, self.steps,
                                self.temperature, self.top_k, self.top_p, self.out_codes,
                                self.frame_kind, self.frame_ws, err_word=self.err, stream=stream)

    def run(self, stream=None, layers: Optional[range] = None, attn_events=None):
        """The whole step.  ``attn_events``: optional list that receives one
        (start, end) CUDA-event pair per paged_decode_attn call, recorded on
        the launch stream."""
        import torch
        L = self.t.layers
        st = stream if stream is not None else torch.cuda.current_stream()
        self._warm = True
        if self.plan_once:
            self.plan(stream=st)
        for l in (layers if layers is not None else range(L)):
            self.append(l, stream=st)
            if attn_events is not None:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(st)
                self.attend(l, stream=st)
                e1.record(st)
                attn_events.append((e0, e1))
            else:
                self.attend(l, stream=st)
        if self.t.logits is not None:
            self.sample(stream=st)
        if self.t.base is not None:
            self.frame(stream=st)

    def capture(self):
        """Capture one whole run() -- every layer's append and attention, the
        sampler and the frame -- as one CUDA graph; replay() then launches
        the step with one call.  The graph reads the buffers this object
        owns, so new inputs are written into them before a replay.  A step
        is run once on a side stream first (outside the capture) unless one
        already ran, so that the library's per-device set-up (kernel
        attributes, the persistent grid size) never happens during capture."""
        import torch
        if not self._warm:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                self.run(stream=side)
            torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        self.graph = g

    def replay(self):
        """One step through the captured graph (on the current stream)."""
        self.graph.replay()

    def capture_attention(self):
        """Capture the attention calls of every layer alone (with plan_once
        the step's plan, then the persistent kernel and merge per layer;
        else planner, persistent kernel and merge per layer) as a second
        graph, to time the attention kernels without host launch gaps.
        Needs a run() (or capture()) first."""
        import torch
        if not self._warm:
            raise RuntimeError("run the step once before capture_attention()")
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            if self.plan_once:
                self.plan()
            for l in range(self.t.layers):
                self.attend(l)
        self.attn_graph = g

    def replay_attention(self):
        """Every layer's attention through the graph of capture_attention()."""
        self.attn_graph.replay()

    def launches_per_step(self) -> int:
        """Kernel launches of one run(): with plan_once one planner, then per
        layer append 1 + attention 2 (persistent kernel, split merge); else
        per layer append 1 + attention 3 (planner too); sampler 2 (chunk
        pass, finish), or 1 for a vocabulary of one 8192-token chunk;
        frame 1."""
        L = self.t.layers
        n = 1 + L * 3 if self.plan_once else L * 4
        if self.t.logits is not None:
            n += 1 if self.t.logits.shape[-1] <= 8192 else 2
        if self.t.base is not None:
            n += 1
        return n


class PrefillStep:
    """One prefill / mixed step of a PrefillBatch: for every layer the
    multi-token append, then causal paged attention of the new tokens.  Owns
    the device copies of the batch description, the outputs and the
    workspace; computes nothing itself."""

    def __init__(self, batch, tensors, device="cuda", with_lse=True):
        import torch
        cfg = batch.cfg
        dev = torch.device(device)
        self.batch, self.cfg, self.t, self.device = batch, cfg, tensors, dev
        i32 = torch.int32
        self.qo_indptr = torch.as_tensor(batch.qo_indptr, dtype=i32).to(dev)
        self.page_table = torch.as_tensor(batch.page_table, dtype=i32).to(dev)
        self.seq_lens = torch.as_tensor(batch.seq_lens, dtype=i32).to(dev)
        self.active = torch.as_tensor(batch.active, dtype=i32).to(dev)
        L = tensors.layers
        T = batch.T
        self.out = torch.empty((L, T, cfg.num_qo_heads, cfg.head_dim), dtype=torch.bfloat16,
                               device=dev)
        self.lse = (torch.empty((L, T, cfg.num_qo_heads), dtype=torch.float32, device=dev)
                    if with_lse else None)
        self.ws = torch.empty(max(B.prefill_workspace_bytes(batch.B), 256), dtype=torch.uint8,
                              device=dev)
        self.err = torch.zeros(1, dtype=i32, device=dev)

    def append(self, layer, stream=None):
        t = self.t
        B.kv_append_tokens(t.cache, layer, t.k[layer], t.v[layer], self.qo_indptr,
                           self.page_table, self.seq_lens, self.active, err_word=self.err,
                           stream=stream)

    def attend(self, layer, stream=None):
        t = self.t
        B.prefill_attn(t.cache, layer, t.q[layer], self.qo_indptr, self.page_table,
                       self.seq_lens, self.active, self.out[layer], self.ws,
                       lse=None if self.lse is None else self.lse[layer], err_word=self.err,
                       stream=stream)

    def run(self, stream=None, attn_events=None):
        import torch
        st = stream if stream is not None else torch.cuda.current_stream()
        for l in range(self.t.layers):
            self.append(l, stream=st)
            if attn_events is not None:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(st)
                self.attend(l, stream=st)
                e1.record(st)
                attn_events.append((e0, e1))
            else:
                self.attend(l, stream=st)

    def launches_per_step(self) -> int:
        """Per layer: the append, the planner and the attention kernel."""
        return 3 * self.t.layers
