#!/usr/bin/env python
"""Benchmark of one batched decode step over a paged KV cache on GB300.

A step is the whole hot path over one batch of synthetic input: for every
layer kv_append + paged_decode_attn, then seeded_sample over the logits
(and, for the frame workload, one frame: a stop/continue sample on channel
0 that gates 12 sequentially sampled codebooks).  Inputs are resident
in HBM when the timed region starts; the per-step KV footprint is far larger
than L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  ``value`` is the step's algorithmic bytes
(KV of every token inside each context + q + out + page-table reads +
appended rows + logits [+ frame rows]) over the step time, in GB/s, summed
over ranks (each rank runs its own replica: "replicas only", weak scaling).
The step is timed as one captured CUDA graph replayed per step (the
production launch; bit-identical to launching the kernels one by one);
``roofline`` times the attention calls of every layer captured alone as a
second graph (CUDA events around its replays), and a third pass launches
the step's kernels one by one (reported under ``eager``).

After the headline workload (long_context by default) the other decode
configurations are measured the same way, with fewer phases, under
``configs``; for each, the oracle runs beside the GPU on the path the bench
times (one more replay of the step graph): ``cpu_baseline`` is its
throughput on a bounded sample and ``parity`` the element-wise comparison,
with the count of sampler near-ties.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

A prefill / mixed-step workload (``--workload mixed_qwen3_4b`` or
``prefill_qwen3_4b_p128``) times instead, per layer, the multi-token append
and the tensor-core causal attention of the step's new tokens, and reports
new tokens/s with the attention kernel's TFLOP/s against the measured bf16
tensor peak.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn HBM GB/s (% of ~8 TB/s) and sampled rows/s at 1 GB300"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------
def step_bytes(batch, cfg, vocab, frame_vocab=0):
    """Algorithmic bytes of the pieces of one step (see the module doc)."""
    act = batch.active.astype(bool)
    n = batch.seq_lens[act].astype(float)
    npg = (n + cfg.page_size - 1) // cfg.page_size
    n_act = int(act.sum())
    kv = float((n * 2 * cfg.num_kv_heads * cfg.head_dim * 2).sum())
    qo = n_act * cfg.num_qo_heads * cfg.head_dim * 2 * 2
    pt = float(npg.sum() * 4)
    attn = kv + qo + pt
    append = n_act * 2 * cfg.num_kv_heads * cfg.head_dim * 2 * 2
    logits = n_act * vocab * 4
    frame = 0
    if cfg.n_codebooks:
        # codebook logits + feedback rows (a frame that stops reads fewer:
        # counted as if none stopped) + the control logits
        frame = (2 * cfg.n_codebooks - 1) * n_act * frame_vocab * 4 + n_act * cfg.ctrl_vocab * 4
    return dict(attn_per_layer=attn, kv_per_layer=kv, append_per_layer=append, logits=logits,
                frame=frame, step=cfg.num_layers * (attn + append) + logits + frame,
                n_active=n_act)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def attn_traffic(workload, source="decode_attn.cu"):
    """DRAM bytes per attention launch (one layer) from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    src = os.path.join(ROOT, "paged_kv_decode_pages_gb300", "csrc", source)
    path = os.path.join(ROOT, "profiles", "attn_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        e = rec.get(workload)
        if e and e.get("source_sha256_16") == h:
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    """nvidia-smi samples of the GPU's clocks and throttle reasons, taken every
    100 ms while started; start() / pause() bracket each timed phase, and
    summary() covers every phase sampled so far."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index, start=True):
        self.proc = None
        self.lines = []
        self.phases = 0
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.sel = str(device_index)
        if start:
            self.start()

    def start(self):
        if self.proc is not None:
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-i", self.sel, "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.phases += 1
        except Exception:
            self.proc = None

    def pause(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines.extend(out.strip().splitlines())
        self.proc = None

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "phases": self.phases}

    def stop(self):
        self.pause()
        return self.summary()


# ---------------------------------------------------------------------------
# the oracle, timed on host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
class OracleRunner:
    """Runs the fp64 oracle over whole layers of the workload (all rows), the
    sampler and the frame, on inputs copied from the device."""

    def __init__(self, batch, tensors):
        import numpy as np
        import oracle
        from paged_kv_decode_pages_gb300 import workloads as W
        self.np, self.oracle, self.W = np, oracle, W
        self.batch, self.t = batch, tensors
        act = batch.active.astype(bool)
        self.rows = [b for b in range(batch.B) if act[b]]
        # compact page table over the active rows: their pages renumbered 1..
        pt = np.zeros_like(batch.page_table)
        self.pages = []
        o = 1
        for b in self.rows:
            k = batch.npages(b)
            pt[b, :k] = np.arange(o, o + k)
            self.pages.extend(batch.page_table[b, :k].tolist())
            o += k
        self.pt = pt
        self.pages_t = None
        self.logits = None if tensors.logits is None else tensors.logits.cpu().numpy()
        self.base = None if tensors.base is None else tensors.base.cpu().numpy()
        self.fb = None if tensors.fb is None else tensors.fb.cpu().numpy()
        self.ctrl = None if tensors.ctrl is None else tensors.ctrl.cpu().numpy()

    def layer_inputs(self, l):
        import torch
        W = self.W
        c = self.t.cache
        if self.pages_t is None:
            self.pages_t = torch.as_tensor(self.pages, dtype=torch.int64, device=c.device)
        body = c[l].index_select(0, self.pages_t).cpu()
        compact = torch.zeros((1, body.shape[0] + 1) + tuple(body.shape[1:]), dtype=body.dtype)
        compact[0, 1:] = body
        return (W.bf16_bits(compact), W.bf16_bits(self.t.q[l]), W.bf16_bits(self.t.k[l]),
                W.bf16_bits(self.t.v[l]))

    def run_layer(self, inputs):
        """One layer's append + attention; returns (seconds, out, lse)."""
        cb, q, k, v = inputs
        b = self.batch
        t0 = time.perf_counter()
        self.oracle.kv_append(cb, 0, k, v, self.pt, b.seq_lens, b.active)
        out, lse, _ = self.oracle.paged_decode_attn(cb, 0, q, self.pt, b.seq_lens, b.active)
        return time.perf_counter() - t0, out, lse

    def run_sampler(self, steps=None):
        """The sampler, then the frame, from the per-slot ``steps`` (default:
        the batch's); returns (seconds, results)."""
        b = self.batch
        t0 = time.perf_counter()
        steps = (b.steps if steps is None else steps).copy()
        res = {}
        if self.logits is not None:
            res["sample"] = self.oracle.seeded_sample(self.logits, b.slots, b.active, b.seeds,
                                                      steps, b.temperature, b.top_k, b.top_p)
        if self.base is not None and self.ctrl is not None:
            res["frame"] = self.oracle.frame_sample(self.ctrl, b.cfg.ctrl_stop, self.base,
                                                    self.fb, b.slots, b.active, b.seeds, steps,
                                                    b.temperature, b.top_k, b.top_p)
        elif self.base is not None:
            res["frame"] = self.oracle.codebook_frame_sample(self.base, self.fb, b.slots,
                                                             b.active, b.seeds, steps,
                                                             b.temperature, b.top_k, b.top_p)
        res["steps"] = steps
        return time.perf_counter() - t0, res


NEAR_TIE = 1e-6  # relative: the top two perturbed scores, or a top-p / min_p cut


def oracle_check(batch, tensors, sizes, step, budget_s=12.0):
    """The oracle beside the GPU on the path the bench times.  One more replay
    of the captured step graph, then the oracle on the same inputs: whole
    layers (every row; as many as fit in about budget_s seconds), the
    sampler over every row and the frame.  Returns (cpu_baseline, parity):
    the oracle's throughput on that sample, and the element-wise comparison
    (attention max-abs / mean-abs, tokens that differ outside and at
    near-ties, with the count of near-ties)."""
    import numpy as np
    import torch
    import oracle
    steps_before = step.steps.cpu().numpy().copy()
    step.out.fill_(float("nan"))
    step.out_tok.fill_(-1)
    if tensors.base is not None:
        step.out_codes.fill_(-9)
    step.replay()
    torch.cuda.synchronize()
    dev_err = int(step.err.item())
    r = OracleRunner(batch, tensors)
    act = batch.active.astype(bool)
    L = batch.cfg.num_layers
    t_total, nbytes, layers = 0.0, 0.0, 0
    amax, asum, acount, lmax = 0.0, 0.0, 0, 0.0
    for l in range(L):
        t, want, want_lse = r.run_layer(r.layer_inputs(l))
        t_total += t
        nbytes += sizes["attn_per_layer"] + sizes["append_per_layer"]
        got = step.out[l].float().cpu().numpy().astype(np.float64)[act]
        e = np.abs(got - want[act])
        amax = max(amax, float(e.max()))
        asum += float(e.sum())
        acount += e.size
        gl = step.lse[l].cpu().numpy().astype(np.float64)[act]
        lmax = max(lmax, float(np.abs(gl - want_lse[act]).max()))
        layers += 1
        if t_total >= budget_s:
            break
    ts, res = r.run_sampler(steps_before)
    t_total += ts
    nbytes += sizes["logits"] + sizes["frame"]
    parity = {"path": "one replay of the captured step graph (the timed path), the slots' "
                      "step counters as that replay read them",
              "device_error_word": dev_err,
              "attn": {"layers": layers, "of_layers": L, "rows": int(act.sum()),
                       "max_abs": amax, "mean_abs": asum / max(acount, 1), "lse_max_abs": lmax,
                       "tolerance": "max-abs 1e-2, mean-abs 1e-3, lse 1e-3",
                       "ok": amax <= 1e-2 and asum / max(acount, 1) <= 1e-3 and lmax <= 1e-3}}
    if "sample" in res:
        tok, _, info, _ = res["sample"]
        got_tok = step.out_tok.cpu().numpy()
        near = ((info["top2_gap_rel"] < NEAR_TIE) | (info["member_margin"] < NEAR_TIE)) & act
        mism = (got_tok != tok) & act
        parity["tokens"] = {"rows": int(act.sum()), "mismatched": int(mism.sum()),
                            "mismatched_outside_near_ties": int((mism & ~near).sum()),
                            "near_ties": int(near.sum()),
                            "near_tie_rule": "top two perturbed scores within 1e-6 relative, "
                                             "or a top-p cut within 1e-6 of p*Z"}
    if "frame" in res:
        codes, _, finfo, _ = res["frame"]
        got = step.out_codes.cpu().numpy()
        n_near = diverge = bad = 0
        for b in np.nonzero(act)[0]:
            for j in range(got.shape[1]):
                nt = finfo[b, j]
                # samplings that ran in both (a stopped row's pad codes have none)
                if got[b, j] == codes[b, j] and codes[b, j] < 0:
                    continue
                tie = nt["top2_gap_rel"] < NEAR_TIE or nt["member_margin"] < NEAR_TIE
                n_near += int(tie)
                if got[b, j] != codes[b, j]:
                    diverge += 1
                    bad += int(not tie)
                    break  # after a near-tie the fed-back codes may legitimately part
        parity["frame"] = {"rows": int(act.sum()), "samplings_per_row": int(got.shape[1]),
                           "rows_diverging": diverge, "diverging_outside_near_ties": bad,
                           "near_ties": n_near}
        parity["steps_match"] = bool(np.array_equal(step.steps.cpu().numpy(), res["steps"]))
    elif "sample" in res:
        parity["steps_match"] = bool(np.array_equal(step.steps.cpu().numpy(), res["steps"]))
    base = {"value": nbytes / t_total / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "%d of %d layers (append + attention, all %d rows) + sampler%s, %.1f s"
                      % (layers, L, batch.B, " + frame" if sizes["frame"] else "", t_total)}
    return base, parity


# ---------------------------------------------------------------------------
# prefill / mixed steps
# ---------------------------------------------------------------------------
PREFILL_METRIC = "prefill / mixed step: new tokens/s and causal-attention TFLOP/s at 1 GB300"


def rank_barrier(world, device):
    """Every rank's device work done, then (N > 1) a barrier over the ranks."""
    import torch
    import torch.distributed as dist
    if device == "cuda":
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()


def rank_max(x, world, device):
    """The maximum of a per-rank time over the ranks (N > 1: one all-reduce
    on a tensor of the process group's device)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replicas_throughput(units_per_rank, world, max_ms):
    """Whole-job throughput of N replicas: all ranks' units over the slowest
    rank's time (units per second)."""
    return world * units_per_rank / (max_ms / 1e3)


def prefill_flops(batch):
    """Algorithmic FLOPs of one layer's attention: every new token of an
    active request, every q head, 2*D for q.k and 2*D for p.v per key of its
    causal range [0, pos]."""
    cfg = batch.cfg
    keys = 0
    for b in range(batch.B):
        if not batch.active[b]:
            continue
        q, n = batch.new_tokens(b), int(batch.seq_lens[b])
        keys += q * (n - q) + q * (q + 1) // 2
    return 4.0 * cfg.head_dim * cfg.num_qo_heads * keys


def tensor_peak(sustained=True):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops_sustained" if sustained else "bf16_tflops"]), "measured"
    except Exception:
        return (1700.0 if sustained else 1900.0), "fallback"


def prefill_cpu_baseline(batch, tensors, budget_s=12.0):
    """The oracle's append + attention on a bounded sample of layer 0: the
    last 32 new tokens of every active request (the rest of the cache as
    drawn), repeated until about budget_s seconds."""
    import numpy as np
    import torch
    import oracle
    from paged_kv_decode_pages_gb300 import workloads as W
    cfg = batch.cfg
    rows = [b for b in range(batch.B) if batch.active[b]]
    pages, o = [], 1
    pt = np.zeros((len(rows), batch.max_pages), np.int32)
    for i, b in enumerate(rows):
        k = (int(batch.seq_lens[b]) + cfg.page_size - 1) // cfg.page_size
        pt[i, :k] = np.arange(o, o + k)
        pages.extend(batch.page_table[b, :k].tolist())
        o += k
    c = tensors.cache[0].index_select(0, torch.as_tensor(pages, device=tensors.cache.device))
    compact = torch.zeros((1, c.shape[0] + 1) + tuple(c.shape[1:]), dtype=c.dtype)
    compact[0, 1:] = c.cpu()
    cb = W.bf16_bits(compact)
    take = [min(32, batch.new_tokens(b)) for b in rows]
    ind = np.concatenate([[0], np.cumsum(take)]).astype(np.int32)
    sel = np.concatenate([np.arange(int(batch.qo_indptr[b + 1]) - k, int(batch.qo_indptr[b + 1]))
                          for b, k in zip(rows, take)])
    selt = torch.as_tensor(sel, device=tensors.q.device)
    q = W.bf16_bits(tensors.q[0].index_select(0, selt))
    k_ = W.bf16_bits(tensors.k[0].index_select(0, selt))
    v_ = W.bf16_bits(tensors.v[0].index_select(0, selt))
    sl = batch.seq_lens[rows].astype(np.int32)
    act = np.ones(len(rows), np.int32)
    flops = 4.0 * cfg.head_dim * cfg.num_qo_heads * sum(
        t * (int(n) - t) + t * (t + 1) // 2 for t, n in zip(take, sl))
    t_total, reps = 0.0, 0
    while t_total < budget_s and reps < 50:
        t0 = time.perf_counter()
        oracle.kv_append_tokens(cb, 0, k_, v_, ind, pt, sl, act)
        oracle.prefill_attn(cb, 0, q, ind, pt, sl, act)
        t_total += time.perf_counter() - t0
        reps += 1
    return {"value": flops * reps / t_total / 1e12, "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "layer 0, the last 32 new tokens of each of %d requests (append + causal "
                      "attention), %d repetitions, %.1f s" % (len(rows), reps, t_total)}


def run_prefill(args, rank, world):
    import numpy as np
    import torch
    import torch.distributed as dist
    import paged_kv_decode_pages_gb300 as pkv
    from paged_kv_decode_pages_gb300 import workloads as W
    from paged_kv_decode_pages_gb300.step import PrefillStep
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pkv.load()
    cfg = W.PREFILL_CONFIGS[args.workload]
    batch = W.make_prefill_batch(cfg)
    tensors = W.PrefillTensors(batch, device="cuda")
    step = PrefillStep(batch, tensors)
    stream = torch.cuda.current_stream()

    def barrier():
        rank_barrier(world, "cuda")

    def max_over_ranks(x):
        return rank_max(x, world, "cuda")

    for _ in range(args.warmup):
        step.run(stream)
    barrier()
    clocks = Clocks(local)
    attn_ev = []
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step.run(stream, attn_events=attn_ev)
    e1.record(stream)
    e1.synchronize()
    clk = clocks.stop()
    total_ms = max_over_ranks(e0.elapsed_time(e1))
    attn_s = float(np.mean([a.elapsed_time(b) for a, b in attn_ev])) / 1e3
    assert int(step.err.item()) == 0, "device error word %#x" % int(step.err.item())
    barrier()

    # end to end: every layer's q, k, v from pinned host memory, the last
    # layer's output back.  Two input sets (the KV cache shared): a copy
    # stream brings step i+1's inputs into one set while step i runs on the
    # other; every copy is inside the timed region.
    from paged_kv_decode_pages_gb300 import workloads as W
    tensors2 = W.PrefillTensors.__new__(W.PrefillTensors)
    tensors2.cache, tensors2.layers = tensors.cache, tensors.layers
    tensors2.q, tensors2.k, tensors2.v = tensors.q.clone(), tensors.k.clone(), tensors.v.clone()
    step2 = PrefillStep(batch, tensors2)
    step2.run(stream)
    pinned = [tensors.q.cpu().pin_memory(), tensors.k.cpu().pin_memory(),
              tensors.v.cpu().pin_memory()]
    sets = [(step, [tensors.q, tensors.k, tensors.v]), (step2, [tensors2.q, tensors2.k, tensors2.v])]
    host_out = torch.empty(step.out[-1].shape, dtype=step.out.dtype, pin_memory=True)
    h2d = sum(h.numel() * h.element_size() for h in pinned)
    d2h = host_out.numel() * host_out.element_size()
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    started = torch.cuda.Event()
    barrier()
    x0 = torch.cuda.Event(enable_timing=True)
    x1 = torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    started.record(stream)
    copy_stream.wait_event(started)

    def copy_in(i):
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(done[i % 2])  # the set's previous step has finished
            for d, h in zip(sets[i % 2][1], pinned):
                d.copy_(h, non_blocking=True)
            copied[i % 2].record(copy_stream)

    copy_in(0)
    for i in range(args.steps):
        if i + 1 < args.steps:
            copy_in(i + 1)
        st_ = sets[i % 2][0]
        stream.wait_event(copied[i % 2])
        st_.run(stream)
        host_out.copy_(st_.out[-1], non_blocking=True)
        done[i % 2].record(stream)
    x1.record(stream)
    x1.synchronize()
    e2e_ms = max_over_ranks(x0.elapsed_time(x1))
    barrier()

    real = int(sum(batch.new_tokens(b) for b in range(batch.B) if batch.active[b]))
    flops = prefill_flops(batch)
    achieved = flops / attn_s / 1e12
    peak, src = tensor_peak(sustained=True)
    line = {
        "metric": PREFILL_METRIC, "value": replicas_throughput(real * args.steps, world, total_ms),
        "unit": "new tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "compute": "bf16 operands, fp32 accumulation in tensor memory (tcgen05)",
        "config": {"workload": cfg.name, "layers": cfg.num_layers, "q_heads": cfg.num_qo_heads,
                   "kv_heads": cfg.num_kv_heads, "head_dim": cfg.head_dim,
                   "page_size": cfg.page_size, "requests": int(batch.active.sum()),
                   "new_tokens": real, "bucket": batch.T,
                   "prompt_requests": int(sum(1 for b in range(batch.B)
                                              if batch.active[b] and batch.new_tokens(b) > 1)),
                   "l2": "inputs larger than L2: %.1f GB of KV across the layers"
                         % (tensors.cache.numel() * 2 / 1e9)},
        "attn": {"us_per_layer": attn_s * 1e6, "tflops": achieved, "flops_per_layer": flops},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": attn_traffic(cfg.name, "prefill_attn.cu"),
                     "kernel": "pkv_prefill_attn (planner + tcgen05 attention kernel), per layer",
                     "peak_source": src + " (bf16, sustained)"},
        "e2e": {"value": replicas_throughput(real * args.steps, world, e2e_ms), "unit": "new tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / args.steps},
        "gpu_launches": step.launches_per_step() * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_baseline(batch, tensors, args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
def make_workload(name, device):
    from paged_kv_decode_pages_gb300 import workloads as W
    cfg = W.CONFIGS[name]
    batch = W.make_batch(cfg)
    tensors = W.Tensors(batch, device=device)
    return cfg, batch, tensors


def workload_config(cfg, batch, l2_note):
    return {"workload": cfg.name, "layers": cfg.num_layers, "q_heads": cfg.num_qo_heads,
            "kv_heads": cfg.num_kv_heads, "head_dim": cfg.head_dim, "page_size": cfg.page_size,
            "batch": batch.B, "active": int(batch.active.sum()),
            "context_min": int(batch.seq_lens[batch.active == 1].min()),
            "context_max": int(batch.seq_lens[batch.active == 1].max()),
            "vocab": cfg.vocab, "temperature": cfg.temperature, "top_k": cfg.top_k,
            "top_p": cfg.top_p, "n_codebooks": cfg.n_codebooks, "l2": l2_note}


def l2_note(cfg, sizes):
    """How the timed inputs relate to L2 (the same string in both arms)."""
    return ("inputs larger than L2: %.1f GB of KV per step"
            % (sizes["kv_per_layer"] * cfg.num_layers / 1e9))


def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores: each step is one whole
    layer of the workload (rotating) plus the sampler."""
    if rank != 0:
        return 0
    import torch
    import oracle
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    cfg, batch, tensors = make_workload(args.workload, dev)
    sizes = step_bytes(batch, cfg, cfg.vocab, cfg.frame_vocab)
    r = OracleRunner(batch, tensors)
    L = cfg.num_layers
    tot, nbytes = 0.0, 0.0
    for i in range(args.warmup + args.steps):
        t = r.run_layer(r.layer_inputs(i % L))[0] + r.run_sampler()[0]
        if i >= args.warmup:
            tot += t
            nbytes += (sizes["attn_per_layer"] + sizes["append_per_layer"] + sizes["logits"]
                       + sizes["frame"])
    value = nbytes / tot / 1e9
    sample = ("per step: 1 of %d layers (append + attention, all %d rows) + sampler%s"
              % (L, batch.B, " + frame" if sizes["frame"] else ""))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, batch, l2_note(cfg, sizes)),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def profile_case(args):
    """A small, self-contained run of one workload for profilers (ncu): the
    full shapes of a configuration with ``--layers`` layers, ``--steps``
    steps, nothing timed.  ``--part sampler`` (or ``frame``) runs only the
    sampler (or the frame) of a decode workload, each step one call; a
    prefill / mixed-step workload runs its append + tensor-core attention
    per layer."""
    import torch
    import paged_kv_decode_pages_gb300 as pkv
    from paged_kv_decode_pages_gb300 import workloads as W
    from paged_kv_decode_pages_gb300.step import DecodeStep, PrefillStep
    pkv.load()
    if args.workload in W.PREFILL_CONFIGS:
        cfg = W.PREFILL_CONFIGS[args.workload]
        batch = W.make_prefill_batch(cfg)
        step = PrefillStep(batch, W.PrefillTensors(batch, device="cuda", layers=args.layers))
        run = step.run
    else:
        cfg = W.CONFIGS[args.workload]
        batch = W.make_batch(cfg)
        step = DecodeStep(batch, W.Tensors(batch, device="cuda", layers=args.layers))
        run = {"all": step.run, "sampler": step.sample, "frame": step.frame}[args.part]
    for _ in range(args.steps):
        run()
    torch.cuda.synchronize()
    err = int(step.err.item())
    print("profile case %s (%s): %d layers x %d steps, err=%d"
          % (cfg.name, args.part, args.layers, args.steps, err))
    return 1 if err else 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long_context")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--configs", default="qwen2_0p5b,llama3_3b,qwen3_4b_frame,tiny",
                    help="further decode workloads measured after the headline one")
    ap.add_argument("--config-cpu-budget", type=float, default=3.0)
    ap.add_argument("--profile-case", action="store_true",
                    help="run a small untimed case for a profiler instead of the bench")
    ap.add_argument("--layers", type=int, default=2, help="layers of the profile case")
    ap.add_argument("--part", default="all", choices=["all", "sampler", "frame"],
                    help="what the profile case runs of a decode workload")
    args = ap.parse_args(argv)
    if args.profile_case:
        return profile_case(args)
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from paged_kv_decode_pages_gb300 import workloads as W
    if args.workload in W.PREFILL_CONFIGS:
        if args.impl == "reference":
            raise SystemExit("the reference arm times the decode step workloads")
        return run_prefill(args, rank, world)
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import torch.distributed as dist
    import paged_kv_decode_pages_gb300 as pkv

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pkv.load()
    clocks = Clocks(local, start=False)
    line, step, rest = measure_decode(args.workload, args, rank, world, local, clocks, full=True)
    lead = rank == 0 and world == 1
    if lead and not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity"] = oracle_check(*rest, step, args.cpu_budget)
    del step, rest
    torch.cuda.empty_cache()
    # the other configurations: kernel figures, a bounded oracle sample and
    # parity each (on rank 0 at N = 1 the oracle legs; every rank times)
    others = [c for c in args.configs.split(",") if c and c != args.workload]
    if others:
        line["configs"] = {}
    for name in others:
        sub, sub_step, sub_rest = measure_decode(name, args, rank, world, local, clocks,
                                                 full=False)
        if lead and not args.no_cpu_baseline:
            sub["cpu_baseline"], sub["parity"] = oracle_check(*sub_rest, sub_step,
                                                              args.config_cpu_budget)
        line["configs"][name] = sub
        del sub_step, sub_rest
        torch.cuda.empty_cache()
    line["clocks"] = clocks.summary()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def measure_decode(name, args, rank, world, local, clocks, full):
    """Times one decode workload.  Every configuration: the step as one
    captured CUDA graph (args.steps replays), the attention calls of every
    layer as a second graph (the roofline), the sampler alone and the frame
    alone.  With full (the headline workload) also the kernel-by-kernel
    pass, the extended sampler and the end-to-end run from pinned host
    memory.  Returns (line, step, (batch, tensors, sizes)); clocks samples
    every timed phase."""
    import numpy as np
    import torch
    from paged_kv_decode_pages_gb300.step import DecodeStep

    cfg, batch, tensors = make_workload(name, "cuda")
    sizes = step_bytes(batch, cfg, cfg.vocab, cfg.frame_vocab)
    step = DecodeStep(batch, tensors)
    stream = torch.cuda.current_stream()

    def barrier():
        rank_barrier(world, "cuda")

    def max_over_ranks(x):
        return rank_max(x, world, "cuda")

    def timed(fn, n):
        """n calls of fn between CUDA events on the launch stream, with the
        clocks sampled; returns the max over ranks of the elapsed ms."""
        barrier()
        clocks.start()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        e1.synchronize()
        clocks.pause()
        ms = max_over_ranks(e0.elapsed_time(e1))
        barrier()
        return ms

    for _ in range(args.warmup):
        step.run(stream)
    barrier()

    # ---- device-resident timed region: the step replayed as one captured
    # CUDA graph (how the pages run a decode step) ------------------------
    step.capture()
    for _ in range(3):
        step.replay()
    total_ms = timed(step.replay, args.steps)

    # ---- the attention kernels alone: the step's plan, then every layer's
    # persistent kernel + merge, captured as one graph, events around K
    # replays (the roofline of the attention kernel) ----------------------
    step.capture_attention()
    for _ in range(3):
        step.replay_attention()
    attn_avg_s = timed(step.replay_attention, args.steps) / 1e3 / (args.steps * cfg.num_layers)

    def per_call_us(fn, n=50, reps=4):
        """fn's kernels captured n times over as one CUDA graph (as they run
        inside the step's graph: no host launch gaps), the graph replayed
        reps times between events; microseconds per call."""
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n):
                fn()
        g.replay()
        return timed(g.replay, reps) / (reps * n) * 1e3

    # ---- sampler alone (rows/s) and frame alone -------------------------
    sampler_us = None
    if tensors.logits is not None:
        sampler_us = per_call_us(lambda: step.sample())
    frame_line = None
    if tensors.base is not None:
        frame_us = per_call_us(lambda: step.frame())
        n_cb = tensors.base.shape[0]
        frame_line = {"us_per_frame": frame_us,
                      "frames_per_s": sizes["n_active"] / (frame_us / 1e6),
                      "samplings_per_frame": n_cb + (1 if tensors.ctrl is not None else 0),
                      "codes_per_s": sizes["n_active"] * n_cb / (frame_us / 1e6)}

    ms_per_step = total_ms / args.steps
    achieved = sizes["attn_per_layer"] / attn_avg_s / 1e9
    peak, peak_src = peaks()
    line = {
        "metric": METRIC,
        "value": replicas_throughput(sizes["step"] * args.steps, world, total_ms) / 1e9,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "compute": "bf16 in, fp32 accumulate (attention); sampler: the fp64 decisions via "
                   "double-float (fp32 pair) sums and an fp32 Gumbel screen, fp64 for contenders",
        "data": "synthetic",
        "config": workload_config(cfg, batch, l2_note(cfg, sizes)),
        "sampled_rows_per_s": world * sizes["n_active"] * args.steps / (total_ms / 1e3),
        "launch": "one captured CUDA graph per step (%d kernels)" % step.launches_per_step(),
        "attn": {"us_per_layer": attn_avg_s * 1e6, "gbs": achieved,
                 "bytes_per_layer": sizes["attn_per_layer"],
                 "timing": "graph of every layer's attention calls, %d replays" % args.steps},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": attn_traffic(cfg.name),
                     "kernel": "pkv_paged_decode_attn_planned (persistent split kernel, "
                               "merge kernel) per layer, with the step's pkv_decode_plan "
                               "amortised over the layers",
                     "peak_source": peak_src},
        "gpu_launches": args.steps * step.launches_per_step(),
    }
    if sampler_us is not None:
        line["sampler"] = {"us_per_call": sampler_us, "timing": "graph of 50 calls, 4 replays",
                           "rows_per_s": sizes["n_active"] / (sampler_us / 1e6),
                           "gbs": sizes["logits"] / (sampler_us / 1e6) / 1e9,
                           "frac": sizes["logits"] / (sampler_us / 1e6) / 1e9 / peak}
    if frame_line:
        line["frame"] = frame_line
    if not full:
        return line, step, (batch, tensors, sizes)

    # ---- the same step launched kernel by kernel, with CUDA events around
    # every attention call -------------------------------------------------
    attn_ev = []
    eager_ms = timed(lambda: step.run(stream, attn_events=attn_ev), args.steps) / args.steps
    attn_ms = [a.elapsed_time(b) for a, b in attn_ev]
    line["eager"] = {"ms_per_step": eager_ms,
                     "value": world * sizes["step"] / (eager_ms / 1e3) / 1e9, "unit": "GB/s",
                     "attn_us_per_call": float(np.mean(attn_ms)) * 1e3,
                     "note": "kernel-by-kernel launches with an event pair around each "
                             "attention call (these events keep the attention from "
                             "overlapping the KV append; on small layers the host's launch "
                             "time shows)"}

    # ---- the sampler with min_p, repetition penalty and log-probs ------
    if tensors.logits is not None:
        ext_set = dict(min_p=0.05, rep_penalty=1.2, rep_window=-1, hist_cap=256)
        step.enable_ext(**ext_set)
        ext_us = per_call_us(lambda: step.sample_ext())
        line["sampler_ext"] = {"us_per_call": ext_us,
                               "rows_per_s": sizes["n_active"] / (ext_us / 1e6),
                               "settings": dict(ext_set, logprobs="raw and processed")}

    # ---- end to end: host (pinned) inputs in, tokens out, every step ----
    # Two copies of the step's input buffers (the KV cache is shared), each
    # with its own captured graph: a copy stream brings step i+1's inputs
    # from pinned host memory into one set while step i runs on the other.
    # Every step's copies and its token read-back are inside the timed
    # region; only the first step's copies are not hidden.
    from paged_kv_decode_pages_gb300 import workloads as W
    tensors2 = W.Tensors.__new__(W.Tensors)
    tensors2.layers, tensors2.cache = tensors.layers, tensors.cache
    for nm in ("q", "k", "v", "logits", "base", "fb", "ctrl"):
        t = getattr(tensors, nm, None)
        setattr(tensors2, nm, None if t is None else (t if nm == "fb" else t.clone()))
    step2 = DecodeStep(batch, tensors2)
    step2.run(stream)
    step2.capture()
    sets = []
    for st_, tn in ((step, tensors), (step2, tensors2)):
        ins = [(tn.q, tensors.q.cpu().pin_memory()), (tn.k, tensors.k.cpu().pin_memory()),
               (tn.v, tensors.v.cpu().pin_memory()),
               (st_.page_table, step.page_table.cpu().pin_memory()),
               (st_.seq_lens, step.seq_lens.cpu().pin_memory()),
               (st_.active, step.active.cpu().pin_memory())]
        for nm in ("logits", "base", "ctrl"):
            if getattr(tn, nm, None) is not None:
                ins.append((getattr(tn, nm), getattr(tensors, nm).cpu().pin_memory()))
        outs = [st_.out_tok, st_.out_kind] + ([st_.out_codes] if tn.base is not None else [])
        sets.append((st_, ins, outs))
    host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in sets[0][2]]
    h2d = sum(h.numel() * h.element_size() for _, h in sets[0][1])
    d2h = sum(h.numel() * h.element_size() for h in host_out)
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    started = torch.cuda.Event()

    def copy_in(i):
        _, ins, _ = sets[i % 2]
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(done[i % 2])  # the set's previous step has finished
            for d, h in ins:
                d.copy_(h, non_blocking=True)
            copied[i % 2].record(copy_stream)

    state = {"i": 0}

    def e2e_step():
        i = state["i"]
        if i == 0:
            started.record(stream)
            copy_stream.wait_event(started)
            copy_in(0)
        if i + 1 < args.steps:
            copy_in(i + 1)
        st_, _, outs = sets[i % 2]
        stream.wait_event(copied[i % 2])
        st_.replay()
        for d, h in zip(outs, host_out):
            h.copy_(d, non_blocking=True)
        done[i % 2].record(stream)
        state["i"] = i + 1

    e2e_ms = timed(e2e_step, args.steps)
    line["e2e"] = {"value": replicas_throughput(sizes["step"] * args.steps, world, e2e_ms) / 1e9,
                   "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                   "ms_per_step": e2e_ms / args.steps}
    del step2, tensors2, sets
    return line, step, (batch, tensors, sizes)


if __name__ == "__main__":
    sys.exit(main())
