"""Batch invariance of the GPU samplers: a request samples the same tokens
whatever batch it lands in ("Adding a Model", vox-serve docs, "How a program
runs").  The same requests (their logits, slot, seed, step and settings) are
placed first, in the middle and last of batches of 1, 5, 32, 64 and 128 rows
among other requests' rows, and every output of theirs -- tokens, kinds,
frame rows, step counters -- must be bit-identical to the request sampled
alone, over several consecutive steps.  Covered: every path of the
seeded sampler (top-k from the chunk candidates, top-p over the whole
vocabulary, the general path for top-k above 512, greedy), the extended
sampler, and both frame entry points."""
import numpy as np
import pytest
import torch

import paged_kv_decode_pages_gb300 as pkv
from paged_kv_decode_pages_gb300 import workloads as W

pytestmark = pytest.mark.gpu

R = 3          # requests under test
FILL0 = R + 1  # first slot of the filler rows (slot 0 is the dummy slot)
N_STEPS = 3


def _u64(a):
    return torch.from_numpy(np.asarray(a, np.uint64).view(np.int64)).view(torch.uint64).cuda()


class Slots:
    """Per-slot sampler state for R requests (slots 1..R) and fillers."""

    def __init__(self, n_slots, T, k, p, seed0):
        rng = np.random.default_rng(seed0)
        self.seeds = rng.integers(0, 2**63, n_slots).astype(np.uint64)
        self.steps = rng.integers(0, 10**6, n_slots).astype(np.int64)
        self.T = np.full(n_slots, T, np.float32)
        self.k = np.full(n_slots, k, np.int32)
        self.p = np.full(n_slots, p, np.float32)

    def dev(self):
        return dict(seeds=_u64(self.seeds), steps=torch.from_numpy(self.steps.copy()).cuda(),
                    T=torch.from_numpy(self.T).cuda(), k=torch.from_numpy(self.k).cuda(),
                    p=torch.from_numpy(self.p).cuda())


def _placement(B, r_rows):
    """Positions of the requests in a batch of B: first, middle, last."""
    if B == 1:
        return [0]
    pos = [0, B // 2, B - 1][: len(r_rows)]
    return pos


def _batch(B, req_logits, fill_rng, V, std, which):
    """Logits [B, V] and slots [B]: request `which[i]` at position pos[i],
    filler rows elsewhere on their own slots."""
    pos = _placement(B, which)
    x = fill_rng.normal(0, std, (B, V)).astype(np.float32)
    slots = FILL0 + np.arange(B, dtype=np.int32)
    for i, r in zip(pos, which):
        x[i] = req_logits[r]
        slots[i] = 1 + r
    return x, slots, pos


SAMPLER_CASES = {
    # long-context sampler: top-p 0.95 over the whole vocabulary, no top-k
    "long_context": dict(V=151936, std=4.0, T=0.7, k=0, p=0.95),
    # Llama-3B sampler: top-k 50 from the chunk candidates, top-p 0.95
    "llama3_3b": dict(V=156940, std=4.0, T=0.6, k=50, p=0.95),
    # Qwen2-0.5B sampler: one chunk per row
    "qwen2_0p5b": dict(V=6561, std=3.0, T=1.0, k=25, p=0.8),
    # the general path: top-k above the 512 candidates
    "general_topk700": dict(V=40000, std=1.0, T=1.0, k=700, p=0.99),
    # greedy
    "greedy": dict(V=32000, std=2.0, T=0.0, k=0, p=1.0),
}


def _run_sampler(x, slots, st, ext=None):
    B, V = x.shape
    dev = torch.from_numpy(x).cuda()
    sl = torch.from_numpy(slots).cuda()
    act = torch.ones(B, dtype=torch.int32, device="cuda")
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    kind = torch.empty(B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stops = torch.tensor([1, 2, 3], dtype=torch.int32, device="cuda")
    if ext is None:
        ws = torch.empty(pkv.sample_workspace_bytes(B, V), dtype=torch.uint8, device="cuda")
        pkv.seeded_sample(dev, sl, act, st["seeds"], st["steps"], st["T"], st["k"], st["p"], tok,
                          kind, ws, salt=4, stop_tokens=stops, audio_lo=100, audio_hi=5000,
                          err_word=err)
        lp = None
    else:
        ws = torch.empty(pkv.sample_ext_workspace_bytes(B, V), dtype=torch.uint8, device="cuda")
        lr = torch.empty(B, dtype=torch.float32, device="cuda")
        lq = torch.empty(B, dtype=torch.float32, device="cuda")
        pkv.seeded_sample_ext(dev, sl, act, st["seeds"], st["steps"], st["T"], st["k"], st["p"],
                              tok, kind, ws, min_p=ext["min_p"], rep_penalty=ext["pen"],
                              rep_window=ext["win"], history=ext["hist"], hist_len=ext["hlen"],
                              logprob_raw=lr, logprob_proc=lq, salt=4, stop_tokens=stops,
                              audio_lo=100, audio_hi=5000, err_word=err)
        lp = (lr, lq)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return tok, kind, lp


def _invariance(case, batches, use_ext=False):
    V, std = case["V"], case["std"]
    rng = np.random.default_rng(V + case["k"])
    req = rng.normal(0, std, (R, V)).astype(np.float32)
    n_slots = FILL0 + max(batches)
    state = Slots(n_slots, case["T"], case["k"], case["p"], seed0=V)
    results = {}
    for B in batches:
        st = state.dev()
        ext = None
        if use_ext:
            hr = np.random.default_rng(5)
            ext = dict(min_p=torch.full((n_slots,), 0.05, device="cuda"),
                       pen=torch.full((n_slots,), 1.2, device="cuda"),
                       win=torch.full((n_slots,), 64, dtype=torch.int32, device="cuda"),
                       hist=torch.from_numpy(hr.integers(0, V, (n_slots, 128)).astype(
                           np.int32)).cuda(),
                       hlen=torch.full((n_slots,), 100, dtype=torch.int32, device="cuda"))
        # B == 1: each request alone; else all of them in one batch
        groups = [[r] for r in range(R)] if B == 1 else [list(range(R))]
        out = {r: [] for r in range(R)}
        for g in groups:
            fill = np.random.default_rng(B * 7 + g[0])
            for step in range(N_STEPS):
                x, slots, pos = _batch(B, req, fill, V, std, g)
                tok, kind, lp = _run_sampler(x, slots, st, ext)
                for i, r in zip(pos, g):
                    rec = [tok[i:i + 1], kind[i:i + 1]]
                    if lp is not None:
                        rec += [lp[0][i:i + 1], lp[1][i:i + 1]]
                    out[r].append(torch.cat([t.view(torch.int32) for t in rec]).cpu())
        steps = st["steps"][1:FILL0].cpu()
        hist = None if ext is None else (ext["hist"][1:FILL0].cpu(), ext["hlen"][1:FILL0].cpu())
        results[B] = (out, steps, hist)
    ref_out, ref_steps, ref_hist = results[batches[0]]
    assert torch.equal(ref_steps, torch.from_numpy(state.steps[1:FILL0] + N_STEPS))
    for B in batches[1:]:
        out, steps, hist = results[B]
        for r in range(R):
            for s in range(N_STEPS):
                assert torch.equal(out[r][s], ref_out[r][s]), (B, r, s, out[r][s], ref_out[r][s])
        assert torch.equal(steps, ref_steps), B
        if hist is not None:
            assert torch.equal(hist[0], ref_hist[0]) and torch.equal(hist[1], ref_hist[1]), B


@pytest.mark.parametrize("name", list(SAMPLER_CASES))
def test_seeded_sample_is_batch_invariant(name):
    _invariance(SAMPLER_CASES[name], (1, 5, 64, 128))


@pytest.mark.parametrize("name", ["long_context", "llama3_3b"])
def test_seeded_sample_ext_is_batch_invariant(name):
    """min_p, a repetition penalty over each slot's ring and both log-probs:
    the tokens, kinds, log-prob bits, rings and step counters."""
    _invariance(SAMPLER_CASES[name], (1, 5, 64), use_ext=True)


# ---------------------------------------------------------------------------
# Frames
# ---------------------------------------------------------------------------
def _frame_inputs(cfg):
    V, n_cb = cfg.frame_vocab, cfg.n_codebooks
    rng = np.random.default_rng(77)
    base = rng.normal(0, cfg.frame_logit_std, (R, n_cb, V)).astype(np.float32)
    ctrl = rng.normal(0, 1.0, (R, cfg.ctrl_vocab)).astype(np.float32)
    ctrl[:, cfg.ctrl_stop] -= 0.5
    ctrl[0, cfg.ctrl_stop] = -np.inf  # request 0 never stops
    fb = torch.from_numpy(rng.normal(0, 1.0, (n_cb, V, V)).astype(np.float32)).cuda()
    return base, ctrl, fb


def _run_frame(cfg, B, which, base_req, ctrl_req, fb, st, fill, full):
    V, n_cb = cfg.frame_vocab, cfg.n_codebooks
    pos = _placement(B, which)
    base = fill.normal(0, cfg.frame_logit_std, (n_cb, B, V)).astype(np.float32)
    ctrl = fill.normal(0, 1.0, (B, cfg.ctrl_vocab)).astype(np.float32)
    slots = FILL0 + np.arange(B, dtype=np.int32)
    for i, r in zip(pos, which):
        base[:, i] = base_req[r]
        ctrl[i] = ctrl_req[r]
        slots[i] = 1 + r
    sl = torch.from_numpy(slots).cuda()
    act = torch.ones(B, dtype=torch.int32, device="cuda")
    kind = torch.empty(B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if full:
        rows = torch.empty((B, 1 + n_cb), dtype=torch.int32, device="cuda")
        ws = torch.empty(pkv.frame_sample_workspace_bytes(n_cb, B, V, cfg.ctrl_vocab),
                         dtype=torch.uint8, device="cuda")
        pkv.frame_sample(torch.from_numpy(ctrl).cuda(), cfg.ctrl_stop,
                         torch.from_numpy(base).cuda(), fb, sl, act, st["seeds"], st["steps"],
                         st["T"], st["k"], st["p"], rows, kind, ws, err_word=err)
    else:
        rows = torch.empty((B, n_cb), dtype=torch.int32, device="cuda")
        ws = torch.empty(pkv.frame_workspace_bytes(n_cb, B, V), dtype=torch.uint8, device="cuda")
        pkv.codebook_frame_sample(torch.from_numpy(base).cuda(), fb, sl, act, st["seeds"],
                                  st["steps"], st["T"], st["k"], st["p"], rows, kind, ws,
                                  err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return {r: torch.cat([rows[i], kind[i:i + 1]]).cpu() for i, r in zip(pos, which)}


@pytest.mark.parametrize("full", [False, True], ids=["codebook_frame", "frame_with_stop"])
def test_frames_are_batch_invariant(full):
    cfg = W.CONFIGS["qwen3_4b_frame"]
    base_req, ctrl_req, fb = _frame_inputs(cfg)
    batches = (1, 5, 32, 64)
    n_slots = FILL0 + max(batches)
    state = Slots(n_slots, cfg.temperature, cfg.top_k, cfg.top_p, seed0=3)
    results = {}
    for B in batches:
        st = state.dev()
        groups = [[r] for r in range(R)] if B == 1 else [list(range(R))]
        out = {r: [] for r in range(R)}
        for g in groups:
            fill = np.random.default_rng(B * 11 + g[0])
            for _ in range(N_STEPS):
                for r, v in _run_frame(cfg, B, g, base_req, ctrl_req, fb, st, fill, full).items():
                    out[r].append(v)
        results[B] = (out, st["steps"][1:FILL0].cpu())
    ref, ref_steps = results[1]
    assert torch.equal(ref_steps, torch.from_numpy(state.steps[1:FILL0] + N_STEPS))
    for B in batches[1:]:
        out, steps = results[B]
        for r in range(R):
            for s in range(N_STEPS):
                assert torch.equal(out[r][s], ref[r][s]), (B, r, s, out[r][s], ref[r][s])
        assert torch.equal(steps, ref_steps), B
