"""pkv_paged_decode_attn_static: the attention entry point for callers that
cannot lend the library any device scratch (a plugin whose host framework
exposes no device allocator, or a serving engine that reserves all device
memory at start-up and allows no allocation later).  It must give the same
bits as pkv_paged_decode_attn with a caller workspace, call after call,
although every call reuses the one scratch array the library keeps on the
device; and it must refuse problems larger than that array.

This file is collected last on purpose, so that in a run of the whole suite
it follows every other GPU test in the same process.  One test here also runs
the call-after-call test again in a fresh Python process, where the first
static call of the process does the per-context set-up."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_pages_gb300 as pkv
from paged_kv_decode_pages_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# the tolerances of the attention parity tests against the oracle
MAX_ABS, MEAN_ABS, LSE_ABS = 1e-2, 1e-3, 1e-3


def _inputs(cfg, layers=None):
    batch = W.make_batch(cfg)
    host = W.Tensors(batch, device="cpu", layers=layers, with_logits=False, with_frame=False)
    dev = dict(cache=host.cache.cuda(), q=host.q.cuda(), k=host.k.cuda(), v=host.v.cuda(),
               pt=torch.from_numpy(batch.page_table).cuda(),
               seq=torch.from_numpy(batch.seq_lens).cuda(),
               act=torch.from_numpy(batch.active).cuda())
    return batch, host, dev


def _both(cfg, layers=None):
    """Every layer: append, then the workspace entry point and the static one
    on the same inputs; the two must agree bit for bit.  Returns the inputs
    and the static call's last outputs."""
    batch, host, d = _inputs(cfg, layers)
    B = batch.B
    Hq, D = cfg.num_qo_heads, cfg.head_dim
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.decode_workspace_bytes(B, Hq, D, batch.max_pages), dtype=torch.uint8,
                     device="cuda")
    want = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    want_lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    got = torch.empty_like(want)
    got_lse = torch.empty_like(want_lse)
    for layer in range(host.layers):
        pkv.kv_append(d["cache"], layer, d["k"][layer], d["v"][layer], d["pt"], d["seq"], d["act"],
                      err_word=err)
        pkv.paged_decode_attn(d["cache"], layer, d["q"][layer], d["pt"], d["seq"], d["act"], want,
                              ws, lse=want_lse, err_word=err)
        got.fill_(float("nan"))
        got_lse.fill_(float("nan"))
        pkv.paged_decode_attn_static(d["cache"], layer, d["q"][layer], d["pt"], d["seq"], d["act"],
                                     got, lse=got_lse, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(got.view(torch.int32), want.view(torch.int32)), layer
        assert torch.equal(got_lse.view(torch.int32), want_lse.view(torch.int32)), layer
    return batch, host, d, got, got_lse


def test_static_scratch_matches_the_workspace_entry_point_call_after_call():
    # first call: long-context shape, several splits per row, padding rows
    first = W.small_variant(W.CONFIGS["long_context"], n_active=3, n_pad=2, ctx_hi=3000,
                            layers=1).replace(ctx_lo=1700)
    # second call on the same scratch: another head layout and other lengths
    second = W.small_variant(W.CONFIGS["qwen2_0p5b"], n_active=9, ctx_hi=1500, layers=1)
    _both(first)
    _both(second)


def test_static_scratch_near_its_limit_matches_the_oracle():
    """The long-context batch at full size (16 rows, 8 of them padding, 2048
    pages a row) needs between 16 and 32 MiB of scratch: bit-equal to the
    workspace entry point on one layer, and two rows against the oracle."""
    cfg = W.CONFIGS["long_context"]
    batch = W.make_batch(cfg)
    need = pkv.decode_workspace_bytes(batch.B, cfg.num_qo_heads, cfg.head_dim, batch.max_pages)
    assert 16 << 20 < need <= pkv._binding.STATIC_SCRATCH_BYTES, need
    batch, host, d, got, got_lse = _both(cfg, layers=1)
    cache_bits = W.bf16_bits(host.cache)
    oracle.kv_append(cache_bits, 0, W.bf16_bits(host.k[0]), W.bf16_bits(host.v[0]),
                     batch.page_table, batch.seq_lens, batch.active)
    rows = [0, int(np.argmax(batch.seq_lens[: cfg.n_active]))]
    only = np.zeros_like(batch.active)
    only[rows] = 1
    want, want_lse, bad = oracle.paged_decode_attn(cache_bits, 0, W.bf16_bits(host.q[0]),
                                                   batch.page_table, batch.seq_lens, only)
    assert bad == 0
    g = got.cpu().numpy().astype(np.float64)[rows]
    e = np.abs(g - want[rows])
    assert e.max() <= MAX_ABS and e.mean() <= MEAN_ABS, (e.max(), e.mean())
    lse = got_lse.cpu().numpy().astype(np.float64)[rows]
    assert np.abs(lse - want_lse[rows]).max() <= LSE_ABS


def test_static_scratch_refuses_problems_larger_than_the_array():
    B, Hq, D, max_pages = 64, 64, 128, 8192
    assert pkv.decode_workspace_bytes(B, Hq, D, max_pages) > pkv._binding.STATIC_SCRATCH_BYTES
    cache = torch.zeros((1, 2, 2, 16, 8, D), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    pt = torch.zeros((B, max_pages), dtype=torch.int32, device="cuda")
    seq = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attn_static(cache, 0, q, pt, seq, seq, out)
    assert e.value.status == 4  # PKV_ERR_WORKSPACE


def test_static_scratch_in_a_fresh_process():
    """The call-after-call test again in a new process: there the static
    entry point's first call makes the per-context address lookup."""
    if os.environ.get("PKV_NO_ALLOC_CHILD"):
        pytest.skip("already the child process")
    env = dict(os.environ, PKV_NO_ALLOC_CHILD="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.abspath(__file__), "-k", "call_after_call"],
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))), env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "1 passed" in r.stdout, r.stdout[-2000:]
