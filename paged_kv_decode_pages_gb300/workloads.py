"""Seeded synthetic inputs for the paged-KV decode step.

This module only draws inputs: it holds none of the step's arithmetic, and it
is the one module that both the CUDA path's tests and the oracle's tests read
inputs from.  Everything is synthetic (there are no trained weights and no
datasets on this path); shapes, value distributions and length mixes follow
the five model-shaped configurations below.

Cache layout (from "Adding a Model", vox-serve docs, section "1. The model
code"): one bf16 tensor [num_layers, num_pages, 2, page_size, num_kv_heads,
head_dim] for all layers; index 0 of dim 2 holds K, index 1 holds V.  Page 0
and slot 0 are the dummy page / dummy slot that padding entries point at
(section "How a program runs"); no request owns them.

Recipe:
  * contexts (seq_len after the append) and page permutations:
    ``numpy.random.default_rng(2000 + config index)``;
  * cache, q, k, v ~ N(0, 1) bf16, logits ~ N(0, sigma^2) fp32, frame
    base ~ N(0, sigma^2), frame feedback ~ N(0, 1), frame control logits
    ~ N(0, sigma_c^2) with ``ctrl_stop_bias`` added to the stop token's:
    ``torch.Generator`` seeded 1000 + config index (Tiny: 0), drawn in a
    fixed order;
  * request r of config c samples with seed 10000 * c + r (Tiny: r), at step 0;
  * pages are handed out from page 1 in row order, contiguously, or as a
    random permutation of 1..P-1 for the Llama-3.2-3B shape;
  * padding rows sit at the end of the batch: active 0, slot 0, seq_len 1,
    page-table row all zeros.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence, Tuple

import numpy as np

KIND_OTHER, KIND_AUDIO, KIND_STOP = 0, 1, 2


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    index: int
    num_layers: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    n_active: int
    n_pad: int
    ctx: Optional[Sequence[int]] = None   # explicit contexts (Tiny)
    ctx_lo: int = 0                       # else uniform integers in [lo, hi]
    ctx_hi: int = 0
    shuffle_pages: bool = False
    vocab: int = 1024
    logit_std: float = 1.0
    temperature: float = 1.0
    top_k: int = 0
    top_p: float = 1.0
    n_codebooks: int = 0                  # > 0: the step ends with a codebook frame
    frame_vocab: int = 0
    frame_logit_std: float = 0.0
    ctrl_vocab: int = 0                   # > 0: the frame opens with a stop/continue sample
    ctrl_stop: int = 1                    # the control token that means stop
    ctrl_logit_std: float = 1.0
    ctrl_stop_bias: float = 0.0

    @property
    def batch(self) -> int:
        return self.n_active + self.n_pad

    @property
    def group(self) -> int:
        return self.num_qo_heads // self.num_kv_heads

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": Config(
        name="tiny", index=0, num_layers=1, num_qo_heads=8, num_kv_heads=2, head_dim=64,
        page_size=16, n_active=4, n_pad=1, ctx=(1, 17, 64, 200), vocab=1024, logit_std=2.0,
        temperature=0.8, top_k=20, top_p=0.9),
    "qwen2_0p5b": Config(
        name="qwen2_0p5b", index=1, num_layers=24, num_qo_heads=14, num_kv_heads=2,
        head_dim=64, page_size=16, n_active=64, n_pad=0, ctx_lo=64, ctx_hi=2048, vocab=6561,
        logit_std=3.0, temperature=1.0, top_k=25, top_p=0.8),
    "llama3_3b": Config(
        name="llama3_3b", index=2, num_layers=28, num_qo_heads=24, num_kv_heads=8,
        head_dim=128, page_size=16, n_active=128, n_pad=0, ctx_lo=512, ctx_hi=4096,
        shuffle_pages=True, vocab=156940, logit_std=4.0, temperature=0.6, top_k=50,
        top_p=0.95),
    "qwen3_4b_frame": Config(
        name="qwen3_4b_frame", index=3, num_layers=36, num_qo_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, n_active=32, n_pad=0, ctx_lo=256, ctx_hi=8192,
        vocab=1024, logit_std=3.0, temperature=0.9, top_k=40, top_p=0.9, n_codebooks=12,
        frame_vocab=1024, frame_logit_std=3.0, ctrl_vocab=2, ctrl_stop=1, ctrl_logit_std=1.0,
        ctrl_stop_bias=-2.0),
    "long_context": Config(
        name="long_context", index=4, num_layers=36, num_qo_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, n_active=8, n_pad=8, ctx_lo=16384, ctx_hi=32768,
        vocab=151936, logit_std=4.0, temperature=0.7, top_k=0, top_p=0.95),
    # the long-context step on a pool of 128-token pages handed out in a
    # random order (the page size of mstar's KV pools)
    "long_context_p128": Config(
        name="long_context_p128", index=5, num_layers=36, num_qo_heads=32, num_kv_heads=8,
        head_dim=128, page_size=128, n_active=8, n_pad=8, ctx_lo=16384, ctx_hi=32768,
        shuffle_pages=True, vocab=151936, logit_std=4.0, temperature=0.7, top_k=0,
        top_p=0.95),
}


@dataclasses.dataclass
class Batch:
    """Host-side (numpy) description of one decode batch."""
    cfg: Config
    seq_lens: np.ndarray      # int32 [B]  (after the append)
    active: np.ndarray        # int32 [B]
    page_table: np.ndarray    # int32 [B, max_pages]
    num_pages: int
    slots: np.ndarray         # int32 [B]
    num_slots: int
    seeds: np.ndarray         # uint64 [num_slots]
    steps: np.ndarray         # int64 [num_slots]
    temperature: np.ndarray   # float32 [num_slots]
    top_k: np.ndarray         # int32 [num_slots]
    top_p: np.ndarray         # float32 [num_slots]

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    def npages(self, b: int) -> int:
        ps = self.cfg.page_size
        return (int(self.seq_lens[b]) + ps - 1) // ps


def make_batch(cfg: Config, max_pages: Optional[int] = None) -> Batch:
    ps = cfg.page_size
    rng = np.random.default_rng(2000 + cfg.index)
    if cfg.ctx is not None:
        ctx = np.asarray(cfg.ctx, dtype=np.int64)
        assert ctx.shape[0] == cfg.n_active
    else:
        ctx = rng.integers(cfg.ctx_lo, cfg.ctx_hi + 1, size=cfg.n_active, dtype=np.int64)
    B = cfg.batch
    seq_lens = np.ones(B, np.int32)
    seq_lens[: cfg.n_active] = ctx
    active = np.zeros(B, np.int32)
    active[: cfg.n_active] = 1
    npg = [(int(n) + ps - 1) // ps for n in ctx]
    mp_needed = max(npg) if npg else 1
    if max_pages is None:
        hi = max(int(ctx.max()) if ctx.size else 1, cfg.ctx_hi)
        max_pages = max((hi + ps - 1) // ps, mp_needed)
    assert max_pages >= mp_needed
    total = int(sum(npg))
    num_pages = total + 1
    ids = np.arange(1, num_pages, dtype=np.int64)
    if cfg.shuffle_pages:
        ids = rng.permutation(ids)
    page_table = np.zeros((B, max_pages), np.int32)
    o = 0
    for b, n in enumerate(npg):
        page_table[b, :n] = ids[o:o + n]
        o += n
    slots = np.zeros(B, np.int32)
    slots[: cfg.n_active] = np.arange(1, cfg.n_active + 1, dtype=np.int32)
    num_slots = cfg.n_active + 1
    seeds = np.zeros(num_slots, np.uint64)
    base_seed = 0 if cfg.index == 0 else 10000 * cfg.index
    for b in range(cfg.n_active):
        seeds[slots[b]] = base_seed + b
    seeds[0] = base_seed + cfg.n_active  # the dummy slot's seed (never drawn from)
    steps = np.zeros(num_slots, np.int64)
    temperature = np.full(num_slots, cfg.temperature, np.float32)
    top_k = np.full(num_slots, cfg.top_k, np.int32)
    top_p = np.full(num_slots, cfg.top_p, np.float32)
    return Batch(cfg, seq_lens, active, page_table, num_pages, slots, num_slots, seeds, steps,
                 temperature, top_k, top_p)


def data_seed(cfg: Config) -> int:
    return 0 if cfg.index == 0 else 1000 + cfg.index


class Tensors:
    """torch tensors of one workload, drawn on ``device`` in a fixed order:
    cache (layer by layer), then for every layer q, k, v, then logits, then
    the frame's base logits and feedback table."""

    def __init__(self, batch: Batch, device="cpu", layers: Optional[int] = None,
                 with_logits: bool = True, with_frame: Optional[bool] = None):
        import torch
        cfg = batch.cfg
        L = cfg.num_layers if layers is None else layers
        B = batch.B
        g = torch.Generator(device=device)
        g.manual_seed(data_seed(cfg))
        bf = torch.bfloat16
        shape = (L, batch.num_pages, 2, cfg.page_size, cfg.num_kv_heads, cfg.head_dim)
        self.cache = torch.empty(shape, dtype=bf, device=device)
        for l in range(L):
            self.cache[l].normal_(0.0, 1.0, generator=g)
        self.q = torch.empty((L, B, cfg.num_qo_heads, cfg.head_dim), dtype=bf, device=device)
        self.k = torch.empty((L, B, cfg.num_kv_heads, cfg.head_dim), dtype=bf, device=device)
        self.v = torch.empty((L, B, cfg.num_kv_heads, cfg.head_dim), dtype=bf, device=device)
        for l in range(L):
            self.q[l].normal_(0.0, 1.0, generator=g)
            self.k[l].normal_(0.0, 1.0, generator=g)
            self.v[l].normal_(0.0, 1.0, generator=g)
        self.logits = None
        if with_logits:
            self.logits = torch.empty((B, cfg.vocab), dtype=torch.float32, device=device)
            self.logits.normal_(0.0, cfg.logit_std, generator=g)
        if with_frame is None:
            with_frame = cfg.n_codebooks > 0
        self.base = self.fb = self.ctrl = None
        if with_frame and cfg.n_codebooks > 0:
            Vf = cfg.frame_vocab
            self.base = torch.empty((cfg.n_codebooks, B, Vf), dtype=torch.float32, device=device)
            self.base.normal_(0.0, cfg.frame_logit_std, generator=g)
            self.fb = torch.empty((cfg.n_codebooks, Vf, Vf), dtype=torch.float32, device=device)
            self.fb.normal_(0.0, 1.0, generator=g)
            if cfg.ctrl_vocab > 0:
                self.ctrl = torch.empty((B, cfg.ctrl_vocab), dtype=torch.float32, device=device)
                self.ctrl.normal_(0.0, cfg.ctrl_logit_std, generator=g)
                self.ctrl[:, cfg.ctrl_stop] += cfg.ctrl_stop_bias
        self.layers = L


# --------------------------------------------------------------------------
# Prefill / mixed steps ("Adding a Model", "How a program runs": prompt rows
# in row buckets; "Supported Models", Qwen3.5 / Qwen3.8 notes: text prefill
# and mixed steps replayed by total tokens on a ladder of buckets)
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    """Request b brings new_b tokens after prefix_b cached ones (a decode row
    is new_b = 1).  Either ``reqs`` lists (prefix, new) pairs, or n_prefill
    prompt requests draw prefix ~ U{prefix_lo..prefix_hi} and new ~
    U{new_lo..new_hi} and n_decode decode rows draw a context ~
    U{ctx_lo..ctx_hi} (prefix = context - 1).  The packed token count is
    padded up to the next bucket of LADDER by one padding request (active 0)
    at the end."""
    name: str
    index: int
    num_layers: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    reqs: Optional[Sequence[Tuple[int, int]]] = None
    n_prefill: int = 0
    prefix_lo: int = 0
    prefix_hi: int = 0
    new_lo: int = 1
    new_hi: int = 1
    n_decode: int = 0
    ctx_lo: int = 1
    ctx_hi: int = 1
    bucket: bool = True
    shuffle_pages: bool = False

    @property
    def group(self) -> int:
        return self.num_qo_heads // self.num_kv_heads

    def replace(self, **kw) -> "PrefillConfig":
        return dataclasses.replace(self, **kw)


PREFILL_CONFIGS = {
    # small enough for the oracle: empty and long prefixes, 1-token decode
    # rows, tiles cut by the ragged tails
    "prefill_tiny": PrefillConfig(
        name="prefill_tiny", index=20, num_layers=1, num_qo_heads=8, num_kv_heads=2,
        head_dim=64, page_size=16,
        reqs=((0, 1), (0, 17), (5, 40), (30, 1), (100, 130), (0, 57), (257, 4))),
    # a mixed step of the Qwen3-4B shape: 4 prompts (up to 4k cached tokens,
    # 0.5-2k new ones) beside 28 decode rows
    "mixed_qwen3_4b": PrefillConfig(
        name="mixed_qwen3_4b", index=21, num_layers=36, num_qo_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, n_prefill=4, prefix_lo=0, prefix_hi=4096, new_lo=512,
        new_hi=2048, n_decode=28, ctx_lo=256, ctx_hi=8192),
    # a text prefill of 8 whole 2k prompts, 128-token pages (mstar's pools)
    "prefill_qwen3_4b_p128": PrefillConfig(
        name="prefill_qwen3_4b_p128", index=22, num_layers=36, num_qo_heads=32,
        num_kv_heads=8, head_dim=128, page_size=128, n_prefill=8, prefix_lo=0, prefix_hi=0,
        new_lo=2048, new_hi=2048, shuffle_pages=True),
}


@dataclasses.dataclass
class PrefillBatch:
    cfg: PrefillConfig
    qo_indptr: np.ndarray     # int32 [B + 1]
    seq_lens: np.ndarray      # int32 [B]  (after the append)
    active: np.ndarray        # int32 [B]
    page_table: np.ndarray    # int32 [B, max_pages]
    num_pages: int

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.qo_indptr[-1])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    def new_tokens(self, b: int) -> int:
        return int(self.qo_indptr[b + 1] - self.qo_indptr[b])


# token buckets of captured prefill / mixed steps: powers of two from 32 to
# 8192 plus 2176, 4352 and 8704 (a step past the last one runs unpadded)
LADDER = tuple(sorted([32 << i for i in range(9)] + [2176, 4352, 8704]))


def ladder_bucket(n: int) -> int:
    """The smallest bucket of the ladder >= n (n itself past the ladder)."""
    for b in LADDER:
        if b >= n:
            return b
    return n


def make_prefill_batch(cfg: PrefillConfig) -> PrefillBatch:
    ps = cfg.page_size
    rng = np.random.default_rng(2000 + cfg.index)
    if cfg.reqs is not None:
        reqs = [(int(a), int(b)) for a, b in cfg.reqs]
    else:
        reqs = []
        for _ in range(cfg.n_prefill):
            reqs.append((int(rng.integers(cfg.prefix_lo, cfg.prefix_hi + 1)),
                         int(rng.integers(cfg.new_lo, cfg.new_hi + 1))))
        for _ in range(cfg.n_decode):
            reqs.append((int(rng.integers(cfg.ctx_lo, cfg.ctx_hi + 1)) - 1, 1))
    T_real = sum(q for _, q in reqs)
    T = ladder_bucket(T_real) if cfg.bucket else T_real
    pad = T - T_real
    B = len(reqs) + (1 if pad > 0 else 0)
    qo = np.zeros(B + 1, np.int32)
    seq = np.ones(B, np.int32)
    act = np.zeros(B, np.int32)
    for b, (pre, q) in enumerate(reqs):
        qo[b + 1] = qo[b] + q
        seq[b] = pre + q
        act[b] = 1
    if pad > 0:
        qo[B] = qo[B - 1] + pad
        seq[B - 1] = pad
    npg = [(int(seq[b]) + ps - 1) // ps for b in range(len(reqs))]
    max_pages = max(npg + [1])
    num_pages = int(sum(npg)) + 1
    ids = np.arange(1, num_pages, dtype=np.int64)
    if cfg.shuffle_pages:
        ids = rng.permutation(ids)
    pt = np.zeros((B, max_pages), np.int32)
    o = 0
    for b, n in enumerate(npg):
        pt[b, :n] = ids[o:o + n]
        o += n
    return PrefillBatch(cfg, qo, seq, act, pt, num_pages)


class PrefillTensors:
    """cache [L, P, 2, ps, Hkv, D] and per layer q [T, Hq, D], k, v
    [T, Hkv, D], all ~ N(0, 1) bf16, drawn on ``device`` from
    ``torch.Generator(1000 + index)`` in that order (cache layer by layer,
    then q, k, v per layer)."""

    def __init__(self, batch: PrefillBatch, device="cpu", layers: Optional[int] = None):
        import torch
        cfg = batch.cfg
        L = cfg.num_layers if layers is None else layers
        g = torch.Generator(device=device)
        g.manual_seed(1000 + cfg.index)
        bf = torch.bfloat16
        shape = (L, batch.num_pages, 2, cfg.page_size, cfg.num_kv_heads, cfg.head_dim)
        self.cache = torch.empty(shape, dtype=bf, device=device)
        for l in range(L):
            self.cache[l].normal_(0.0, 1.0, generator=g)
        T = batch.T
        self.q = torch.empty((L, T, cfg.num_qo_heads, cfg.head_dim), dtype=bf, device=device)
        self.k = torch.empty((L, T, cfg.num_kv_heads, cfg.head_dim), dtype=bf, device=device)
        self.v = torch.empty((L, T, cfg.num_kv_heads, cfg.head_dim), dtype=bf, device=device)
        for l in range(L):
            self.q[l].normal_(0.0, 1.0, generator=g)
            self.k[l].normal_(0.0, 1.0, generator=g)
            self.v[l].normal_(0.0, 1.0, generator=g)
        self.layers = L


def bf16_bits(t) -> np.ndarray:
    """bf16 torch tensor -> numpy uint16 array of its bits (host copy)."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def small_variant(cfg: Config, n_active: int, ctx_hi: int, layers: int = 2,
                  n_pad: Optional[int] = None, vocab: Optional[int] = None) -> Config:
    """The same heads / head_dim / page size / sampler settings at a size the
    oracle finishes in seconds, still spanning several splits and a ragged
    last page."""
    kw = dict(n_active=n_active, num_layers=layers, ctx=None,
              ctx_lo=min(cfg.ctx_lo if cfg.ctx is None else 1, ctx_hi), ctx_hi=ctx_hi,
              name=cfg.name + "_small")
    if n_pad is not None:
        kw["n_pad"] = n_pad
    if vocab is not None:
        kw["vocab"] = vocab
    return cfg.replace(**kw)
