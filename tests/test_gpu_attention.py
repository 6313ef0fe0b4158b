"""GPU parity of kv_append and paged_decode_attn against the fp64 oracle, on
the same seeded inputs (drawn on the CPU, copied to both sides).

Tolerances (bf16 inputs, fp32 accumulation): attention output within
max-abs 1e-2 and mean-abs 1e-3 of the oracle; lse within 1e-3; the append
bit-exact on every byte outside the dummy page 0 (which padding rows may
all write)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_pages_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 1e-2, 1e-3, 1e-3


def _cases():
    C = W.CONFIGS
    return {
        "tiny": C["tiny"],
        "qwen2_small": W.small_variant(C["qwen2_0p5b"], n_active=6, ctx_hi=700, layers=2),
        "llama3_small": W.small_variant(C["llama3_3b"], n_active=5, ctx_hi=1100, layers=2),
        "qwen3_frame_small": W.small_variant(C["qwen3_4b_frame"], n_active=4, ctx_hi=1500,
                                             layers=2),
        "long_small": W.small_variant(C["long_context"], n_active=3, n_pad=3, ctx_hi=2100,
                                      layers=2).replace(ctx_lo=1500),
        # split boundaries: 512 tokens per split, 16 per page
        "edges_d128": W.Config(name="edges_d128", index=7, num_layers=1, num_qo_heads=8,
                               num_kv_heads=2, head_dim=128, page_size=16, n_active=9, n_pad=2,
                               ctx=(1, 15, 16, 17, 511, 512, 513, 528, 1025)),
        "edges_d64_g7": W.Config(name="edges_d64_g7", index=8, num_layers=1, num_qo_heads=14,
                                 num_kv_heads=2, head_dim=64, page_size=16, n_active=6, n_pad=1,
                                 ctx=(1, 16, 33, 512, 513, 800), shuffle_pages=True),
        "g1_mha": W.Config(name="g1_mha", index=9, num_layers=1, num_qo_heads=4, num_kv_heads=4,
                           head_dim=128, page_size=16, n_active=3, n_pad=0, ctx=(5, 600, 40)),
        "g12_two_qblocks": W.Config(name="g12", index=10, num_layers=1, num_qo_heads=24,
                                    num_kv_heads=2, head_dim=128, page_size=16, n_active=3,
                                    n_pad=1, ctx=(7, 700, 1200)),
        # pages of 32, 64 and 128 tokens (the kernels stream 16-token blocks):
        # page and split boundaries, shuffled pools
        "page32_shuffled": W.Config(name="page32", index=12, num_layers=1, num_qo_heads=8,
                                    num_kv_heads=2, head_dim=128, page_size=32, n_active=7,
                                    n_pad=1, ctx=(1, 31, 32, 33, 513, 1100, 48),
                                    shuffle_pages=True),
        "page64_d64_g7": W.Config(name="page64", index=13, num_layers=1, num_qo_heads=14,
                                  num_kv_heads=2, head_dim=64, page_size=64, n_active=5,
                                  n_pad=1, ctx=(63, 64, 65, 512, 700), shuffle_pages=True),
        "page128": W.Config(name="page128", index=14, num_layers=2, num_qo_heads=32,
                            num_kv_heads=8, head_dim=128, page_size=128, n_active=7, n_pad=2,
                            ctx=(1, 127, 128, 129, 513, 2100, 4000), shuffle_pages=True),
        "long_p128_small": W.small_variant(W.CONFIGS["long_context_p128"], n_active=3, n_pad=2,
                                           ctx_hi=2600, layers=2).replace(ctx_lo=1500),
        # every row a whole number of 512-token splits: no short last split
        "whole_splits": W.Config(name="whole", index=16, num_layers=1, num_qo_heads=8,
                                 num_kv_heads=2, head_dim=128, page_size=16, n_active=3,
                                 n_pad=1, ctx=(512, 1024, 2048)),
        # more rows than the kernel's shared-memory split table holds (512):
        # the unit table is read from global memory
        "wide_batch_600": W.Config(name="wide600", index=15, num_layers=1, num_qo_heads=4,
                                   num_kv_heads=2, head_dim=64, page_size=16, n_active=600,
                                   n_pad=24, ctx_lo=1, ctx_hi=1100, shuffle_pages=True),
    }


CASES = _cases()


def _run(cfg, out_fp32):
    from paged_kv_decode_pages_gb300.step import DecodeStep
    batch = W.make_batch(cfg)
    host = W.Tensors(batch, device="cpu", with_logits=False, with_frame=False)
    cache_bits = W.bf16_bits(host.cache)
    dev = W.Tensors.__new__(W.Tensors)
    dev.cache = host.cache.cuda()
    dev.q, dev.k, dev.v = host.q.cuda(), host.k.cuda(), host.v.cuda()
    dev.logits = dev.base = dev.fb = None
    dev.layers = host.layers
    step = DecodeStep(batch, dev, out_fp32=out_fp32)
    step.run()
    torch.cuda.synchronize()
    return batch, host, cache_bits, step


@pytest.mark.parametrize("out_fp32", [True, False])
@pytest.mark.parametrize("name", list(CASES))
def test_append_and_attention_match_oracle(name, out_fp32):
    cfg = CASES[name]
    batch, host, cache_bits, step = _run(cfg, out_fp32)
    assert int(step.err.item()) == 0
    worst = 0.0
    for l in range(host.layers):
        bad = oracle.kv_append(cache_bits, l, W.bf16_bits(host.k[l]), W.bf16_bits(host.v[l]),
                               batch.page_table, batch.seq_lens, batch.active)
        assert bad == 0
        want, want_lse, bad = oracle.paged_decode_attn(cache_bits, l, W.bf16_bits(host.q[l]),
                                                       batch.page_table, batch.seq_lens,
                                                       batch.active)
        assert bad == 0
        got = step.out[l].float().cpu().numpy().astype(np.float64)
        err = np.abs(got - want)
        assert err.max() <= MAX_ABS, (name, l, err.max())
        assert err.mean() <= MEAN_ABS, (name, l, err.mean())
        worst = max(worst, float(err.max()))
        act = batch.active.astype(bool)
        lse = step.lse[l].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(lse[act] - want_lse[act]) <= LSE_ABS)
        assert np.all(np.isneginf(lse[~act]))
        assert np.all(got[~act] == 0.0)
    # every byte of the cache outside page 0 equals the oracle's
    got_cache = W.bf16_bits(step.t.cache)
    np.testing.assert_array_equal(got_cache[:, 1:], cache_bits[:, 1:])
    if out_fp32:
        # fp32 output: far inside the contract (no bf16 rounding of the output)
        assert worst < 1e-4, worst


@pytest.mark.parametrize("name", list(CASES))
def test_planned_calls_equal_per_call_plans(name):
    """One decode_plan for the step, then the planned attention of every
    layer, gives the same bits as each layer's call planning for itself
    (the planned calls after the first rely on the merge resetting the unit
    counter); two more rounds on one new plan give them again."""
    batch, host, cache_bits, step = _run(CASES[name], True)
    assert step.plan_once
    planned = step.out.clone()
    planned_lse = step.lse.clone()
    step.plan_once = False
    for l in range(host.layers):
        step.attend(l)
    torch.cuda.synchronize()
    assert torch.equal(step.out.view(torch.int32), planned.view(torch.int32)), name
    assert torch.equal(step.lse.view(torch.int32), planned_lse.view(torch.int32)), name
    step.plan_once = True
    step.plan()
    for _ in range(2):  # the second round follows planned calls only
        step.out.zero_()
        for l in range(host.layers):
            step.attend(l)
    torch.cuda.synchronize()
    assert torch.equal(step.out.view(torch.int32), planned.view(torch.int32)), name
    assert int(step.err.item()) == 0


def test_single_token_and_identical_keys_closed_forms():
    """n = 1 gives v itself; identical keys give the mean of V."""
    from paged_kv_decode_pages_gb300.step import DecodeStep
    cfg = W.Config(name="closed", index=11, num_layers=1, num_qo_heads=8, num_kv_heads=2,
                   head_dim=128, page_size=16, n_active=2, n_pad=0, ctx=(1, 1000))
    batch = W.make_batch(cfg)
    host = W.Tensors(batch, device="cpu", with_logits=False, with_frame=False)
    # row 1: every key equal to its new key
    n = int(batch.seq_lens[1])
    for t in range(n - 1):
        p = batch.page_table[1, t // 16]
        host.cache[0, p, 0, t % 16] = host.k[0, 1]
    dev = W.Tensors.__new__(W.Tensors)
    dev.cache, dev.q, dev.k, dev.v = host.cache.cuda(), host.q.cuda(), host.k.cuda(), host.v.cuda()
    dev.logits = dev.base = dev.fb = None
    dev.layers = 1
    step = DecodeStep(batch, dev, out_fp32=True)
    step.run()
    out = step.out[0].cpu().double()
    v_new = host.v[0].double()
    for h in range(8):
        assert torch.equal(out[0, h], v_new[0, h // 4])
    # mean of V over row 1 (after the append)
    vs = []
    for t in range(n):
        p = batch.page_table[1, t // 16]
        vs.append(host.v[0, 1] if t == n - 1 else host.cache[0, p, 1, t % 16])
    mean_v = torch.stack(vs).double().mean(0)
    for h in range(8):
        assert torch.allclose(out[1, h], mean_v[h // 4], atol=2e-5, rtol=0)


def test_bad_inputs_set_error_bits_and_spare_other_rows():
    from paged_kv_decode_pages_gb300.step import DecodeStep
    cfg = W.Config(name="bad", index=12, num_layers=1, num_qo_heads=8, num_kv_heads=2,
                   head_dim=64, page_size=16, n_active=4, n_pad=0, ctx=(40, 70, 90, 600))
    batch = W.make_batch(cfg)
    host = W.Tensors(batch, device="cpu", with_logits=False, with_frame=False)
    cache_bits = W.bf16_bits(host.cache)
    batch.page_table[0, 1] = batch.num_pages + 5        # page id out of range (read side)
    batch.page_table[1, (70 - 1) // 16] = -7            # page id out of range (append side)
    batch.seq_lens[2] = batch.max_pages * 16 + 3        # seq_len beyond the page table
    dev = W.Tensors.__new__(W.Tensors)
    dev.cache, dev.q, dev.k, dev.v = host.cache.cuda(), host.q.cuda(), host.k.cuda(), host.v.cuda()
    dev.logits = dev.base = dev.fb = None
    dev.layers = 1
    step = DecodeStep(batch, dev, out_fp32=True)
    step.run()
    torch.cuda.synchronize()
    err = int(step.err.item())
    assert err & 0x1 and err & 0x2  # PKV_DEV_ERR_PAGE, PKV_DEV_ERR_SEQ_LEN
    # row 3 is valid: exact parity; row 2 (bad length) is zeros
    oracle.kv_append(cache_bits, 0, W.bf16_bits(host.k[0]), W.bf16_bits(host.v[0]),
                     batch.page_table, batch.seq_lens, batch.active)
    want, _, _ = oracle.paged_decode_attn(cache_bits, 0, W.bf16_bits(host.q[0]), batch.page_table,
                                          batch.seq_lens, batch.active)
    got = step.out[0].cpu().numpy()
    assert np.abs(got[3] - want[3]).max() < 1e-4
    assert np.all(got[2] == 0)
    # the append wrote nothing for rows 1 (bad page) and 2 (bad length)
    got_cache = W.bf16_bits(step.t.cache)
    np.testing.assert_array_equal(got_cache[:, 1:], cache_bits[:, 1:])


def test_planned_call_on_lengths_changed_after_the_plan_is_reported_and_stays_in_bounds():
    """The planned attention trusts the caller to keep the lengths of the
    plan.  When they change after pkv_decode_plan (row 0 past max_pages, row
    1 exactly max_pages so that its planned last split lies past the end, row
    2 shorter), the call reports PKV_DEV_ERR_SEQ_LEN, writes nothing outside
    its workspace and outputs, and the next plan on correct lengths gives the
    per-call result again."""
    import paged_kv_decode_pages_gb300 as pkv
    cfg = W.Config(name="replan", index=17, num_layers=1, num_qo_heads=8, num_kv_heads=2,
                   head_dim=128, page_size=16, n_active=3, n_pad=1, ctx=(100, 700, 40))
    batch = W.make_batch(cfg, max_pages=64)  # max_tokens 1024: two splits at most
    host = W.Tensors(batch, device="cpu", with_logits=False, with_frame=False)
    cache, q = host.cache.cuda(), host.q[0].cuda()
    pt = torch.from_numpy(batch.page_table).cuda()
    seq = torch.from_numpy(batch.seq_lens).cuda()
    act = torch.from_numpy(batch.active).cuda()
    B, Hq, D = batch.B, cfg.num_qo_heads, cfg.head_dim
    need = pkv.decode_workspace_bytes(B, Hq, D, batch.max_pages)
    guard = 4096
    ws_full = torch.zeros(need + guard, dtype=torch.uint8, device="cuda")
    ws = ws_full[:need]
    ws_full[need:] = 0x5A
    out = torch.zeros((B, Hq, D), dtype=torch.float32, device="cuda")
    lse = torch.zeros((B, Hq), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache_before = cache.clone()

    pkv.decode_plan(cache, Hq, batch.max_pages, seq, act, ws, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    seq_changed = seq.clone()
    seq_changed[0] = batch.max_pages * 16 + 5
    seq_changed[1] = batch.max_pages * 16
    seq_changed[2] = 30
    pkv.paged_decode_attn_planned(cache, 0, q, pt, seq_changed, act, out, ws, lse=lse,
                                  err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x2  # PKV_DEV_ERR_SEQ_LEN
    assert torch.all(ws_full[need:] == 0x5A)
    assert torch.equal(cache, cache_before)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))  # past max_pages
    assert torch.all(out[3] == 0)  # the padding row

    # a new plan on the original lengths: planned = per-call, bit for bit
    err.zero_()
    pkv.decode_plan(cache, Hq, batch.max_pages, seq, act, ws, err_word=err)
    pkv.paged_decode_attn_planned(cache, 0, q, pt, seq, act, out, ws, lse=lse, err_word=err)
    want = torch.empty_like(out)
    want_lse = torch.empty_like(lse)
    pkv.paged_decode_attn(cache, 0, q, pt, seq, act, want, ws, lse=want_lse, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out.view(torch.int32), want.view(torch.int32))
    assert torch.equal(lse.view(torch.int32), want_lse.view(torch.int32))
    assert torch.all(ws_full[need:] == 0x5A)
