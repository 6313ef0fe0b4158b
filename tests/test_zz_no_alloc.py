"""pkv_paged_decode_attn_static: the attention entry point for callers that
cannot lend the library any device scratch (a plugin whose host framework
exposes no device allocator, or a serving engine that reserves all device
memory at start-up and allows no allocation later).  It must give the same
results as pkv_paged_decode_attn with a caller workspace, call after call,
although every call reuses the one scratch array the library keeps on the
device; and it must refuse problems larger than that array.

This file is collected last on purpose: it also runs after every other GPU
test in the same process, and alone in a fresh one."""
import numpy as np
import pytest
import torch

import paged_kv_decode_pages_gb300 as pkv
from paged_kv_decode_pages_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# the tolerances of the attention parity tests
MAX_ABS, MEAN_ABS = 1e-2, 1e-3


def _inputs(cfg):
    batch = W.make_batch(cfg)
    host = W.Tensors(batch, device="cpu", with_logits=False, with_frame=False)
    dev = dict(cache=host.cache.cuda(), q=host.q.cuda(), k=host.k.cuda(), v=host.v.cuda(),
               pt=torch.from_numpy(batch.page_table).cuda(),
               seq=torch.from_numpy(batch.seq_lens).cuda(),
               act=torch.from_numpy(batch.active).cuda())
    return batch, dev


def _both(cfg):
    batch, d = _inputs(cfg)
    B = batch.B
    Hq, D = cfg.num_qo_heads, cfg.head_dim
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.decode_workspace_bytes(B, Hq, D, batch.max_pages), dtype=torch.uint8,
                     device="cuda")
    want = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    want_lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    got = torch.empty_like(want)
    got_lse = torch.empty_like(want_lse)
    for layer in range(cfg.num_layers):
        pkv.kv_append(d["cache"], layer, d["k"][layer], d["v"][layer], d["pt"], d["seq"], d["act"],
                      err_word=err)
        pkv.paged_decode_attn(d["cache"], layer, d["q"][layer], d["pt"], d["seq"], d["act"], want,
                              ws, lse=want_lse, err_word=err)
        pkv.paged_decode_attn_static(d["cache"], layer, d["q"][layer], d["pt"], d["seq"], d["act"],
                                     got, lse=got_lse, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        diff = (got - want).abs()
        assert float(diff.max()) <= MAX_ABS and float(diff.mean()) <= MEAN_ABS
        act = d["act"].bool()
        assert float((got_lse[act] - want_lse[act]).abs().max()) <= 1e-3


def test_static_scratch_matches_the_workspace_entry_point_call_after_call():
    # first call: long-context shape, several splits per row, padding rows
    first = W.small_variant(W.CONFIGS["long_context"], n_active=3, n_pad=2, ctx_hi=3000,
                            layers=1).replace(ctx_lo=1700)
    # second call on the same scratch: another head layout and other lengths
    second = W.small_variant(W.CONFIGS["qwen2_0p5b"], n_active=9, ctx_hi=1500, layers=1)
    _both(first)
    _both(second)


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
