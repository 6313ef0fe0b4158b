"""Pins of the prefill / mixed-step oracle (multi-token append and causal
paged attention; "Adding a Model", "How a program runs": prompt rows in row
buckets; "Supported Models", Qwen3.5 / Qwen3.8 notes: text prefill and
mixed steps) against things other than itself:
  * torch's fp64 scaled_dot_product_attention with an explicit causal mask
    on the densely gathered sequence (GQA by repeat_interleave);
  * with one new token per request it is the (independently pinned) decode
    oracle;
  * closed forms: identical keys give the running mean of the values, an
    empty prefix makes the first token attend only to itself;
  * chunked prefill: a prompt appended and attended in two steps gives
    each token the same output as in one step;
  * the append's bytes against index arithmetic."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_pages_gb300 import workloads as W


def _inputs(cfg):
    batch = W.make_prefill_batch(cfg)
    t = W.PrefillTensors(batch, device="cpu")
    return batch, t


def _dense_reference(cache_bits, layer, q_bits, batch, scale):
    """Gather each request's keys / values densely in fp64 and run torch's
    SDPA with a boolean mask key <= position."""
    L, P, _, ps, Hkv, D = cache_bits.shape
    c = torch.from_numpy(cache_bits.view(np.int16)).view(torch.bfloat16).double()
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).double()
    Hq = q.shape[1]
    G = Hq // Hkv
    out = torch.zeros_like(q)
    for b in range(batch.B):
        nq = batch.new_tokens(b)
        if not batch.active[b] or nq == 0:
            continue
        n = int(batch.seq_lens[b])
        pos = torch.arange(n - nq, n)
        pages = torch.from_numpy(batch.page_table[b, :(n + ps - 1) // ps].astype(np.int64))
        kk = c[layer, pages, 0].reshape(-1, Hkv, D)[:n]  # [n, Hkv, D]
        vv = c[layer, pages, 1].reshape(-1, Hkv, D)[:n]
        qq = q[batch.qo_indptr[b]:batch.qo_indptr[b + 1]]  # [nq, Hq, D]
        kq = kk.permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, n, D]
        vq = vv.permute(1, 0, 2).repeat_interleave(G, dim=0)
        mask = torch.arange(n)[None, :] <= pos[:, None]       # [nq, n]
        o = torch.nn.functional.scaled_dot_product_attention(
            qq.permute(1, 0, 2), kq, vq, attn_mask=mask, scale=scale)
        out[batch.qo_indptr[b]:batch.qo_indptr[b + 1]] = o.permute(1, 0, 2)
    return out.numpy()


CASES = {
    "tiny_g4_d64": W.PREFILL_CONFIGS["prefill_tiny"],
    "g1_d128_p32": W.PrefillConfig(name="g1", index=30, num_layers=1, num_qo_heads=3,
                                   num_kv_heads=3, head_dim=128, page_size=32,
                                   reqs=((0, 33), (40, 1), (7, 70)), shuffle_pages=True),
    "g7_d64_p128": W.PrefillConfig(name="g7", index=31, num_layers=2, num_qo_heads=14,
                                   num_kv_heads=2, head_dim=64, page_size=128,
                                   reqs=((200, 60), (0, 129), (127, 2)), bucket=False),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_oracle_matches_torch_sdpa_with_a_causal_mask(name):
    cfg = CASES[name]
    batch, t = _inputs(cfg)
    cache = W.bf16_bits(t.cache)
    layer = t.layers - 1
    assert oracle.kv_append_tokens(cache, layer, W.bf16_bits(t.k[layer]), W.bf16_bits(t.v[layer]),
                                   batch.qo_indptr, batch.page_table, batch.seq_lens,
                                   batch.active) == 0
    q = W.bf16_bits(t.q[layer])
    scale = 1.0 / np.sqrt(cfg.head_dim)
    out, lse, bad = oracle.prefill_attn(cache, layer, q, batch.qo_indptr, batch.page_table,
                                        batch.seq_lens, batch.active)
    assert bad == 0
    want = _dense_reference(cache, layer, q, batch, scale)
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)
    # padding tokens: zeros, lse -inf
    pad = np.zeros(batch.T, bool)
    for b in range(batch.B):
        if not batch.active[b]:
            pad[batch.qo_indptr[b]:batch.qo_indptr[b + 1]] = True
    assert np.all(out[pad] == 0) and np.all(np.isneginf(lse[pad]))
    assert np.all(np.isfinite(lse[~pad]))


def test_one_new_token_per_request_is_the_decode_oracle():
    cfg = W.PrefillConfig(name="dec", index=32, num_layers=1, num_qo_heads=8, num_kv_heads=2,
                          head_dim=64, page_size=16, reqs=((0, 1), (16, 1), (300, 1), (40, 1)),
                          bucket=False, shuffle_pages=True)
    batch, t = _inputs(cfg)
    cache = W.bf16_bits(t.cache)
    q = W.bf16_bits(t.q[0])
    out, lse, bad = oracle.prefill_attn(cache, 0, q, batch.qo_indptr, batch.page_table,
                                        batch.seq_lens, batch.active)
    dout, dlse, dbad = oracle.paged_decode_attn(cache, 0, q, batch.page_table, batch.seq_lens,
                                                batch.active)
    assert bad == dbad == 0
    np.testing.assert_array_equal(out, dout)
    np.testing.assert_array_equal(lse, dlse)


def test_identical_keys_give_the_running_mean_of_the_values():
    """All keys equal: every allowed key has the same score, so the token at
    position p gets mean(v_0..v_p) -- an off-by-one in the causal range
    changes every row."""
    cfg = W.PrefillConfig(name="mean", index=33, num_layers=1, num_qo_heads=4, num_kv_heads=2,
                          head_dim=64, page_size=16, reqs=((0, 20), (9, 7)), bucket=False)
    batch, t = _inputs(cfg)
    t.cache[:, :, 0] = t.cache[0, 1, 0, 0, 0]  # every K row the same vector
    t.k[:] = t.cache[0, 1, 0, 0, 0]
    cache = W.bf16_bits(t.cache)
    assert oracle.kv_append_tokens(cache, 0, W.bf16_bits(t.k[0]), W.bf16_bits(t.v[0]),
                                   batch.qo_indptr, batch.page_table, batch.seq_lens,
                                   batch.active) == 0
    out, _, _ = oracle.prefill_attn(cache, 0, W.bf16_bits(t.q[0]), batch.qo_indptr,
                                    batch.page_table, batch.seq_lens, batch.active)
    c = torch.from_numpy(cache.view(np.int16)).view(torch.bfloat16).double().numpy()
    for b in range(batch.B):
        n = int(batch.seq_lens[b])
        nq = batch.new_tokens(b)
        vals = np.stack([c[0, batch.page_table[b, j // 16], 1, j % 16] for j in range(n)])
        for i in range(nq):
            p = n - nq + i
            want = vals[:p + 1].mean(axis=0)  # [Hkv, D]
            got = out[batch.qo_indptr[b] + i]  # [Hq, D]
            np.testing.assert_allclose(got, np.repeat(want, 2, axis=0), atol=1e-12)


def test_first_token_of_an_empty_prefix_attends_only_to_itself():
    cfg = W.PrefillConfig(name="first", index=34, num_layers=1, num_qo_heads=4, num_kv_heads=4,
                          head_dim=64, page_size=16, reqs=((0, 5),), bucket=False)
    batch, t = _inputs(cfg)
    cache = W.bf16_bits(t.cache)
    oracle.kv_append_tokens(cache, 0, W.bf16_bits(t.k[0]), W.bf16_bits(t.v[0]), batch.qo_indptr,
                            batch.page_table, batch.seq_lens, batch.active)
    out, lse, _ = oracle.prefill_attn(cache, 0, W.bf16_bits(t.q[0]), batch.qo_indptr,
                                      batch.page_table, batch.seq_lens, batch.active)
    v0 = t.v[0, 0].double().numpy()
    np.testing.assert_array_equal(out[0], v0)
    q0 = t.q[0, 0].double().numpy()
    k0 = t.k[0, 0].double().numpy()
    np.testing.assert_allclose(lse[0], (q0 * k0).sum(-1) / 8.0, atol=1e-12)


def test_chunked_prefill_equals_one_step():
    """A 150-token prompt after a 30-token prefix, attended in one step or as
    64 + 86 tokens in two steps: each token's output is the same."""
    base = dict(num_layers=1, num_qo_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
                bucket=False)
    one = W.PrefillConfig(name="one", index=35, reqs=((30, 150),), **base)
    batch, t = _inputs(one)
    cache1 = W.bf16_bits(t.cache)
    k, v, q = W.bf16_bits(t.k[0]), W.bf16_bits(t.v[0]), W.bf16_bits(t.q[0])
    oracle.kv_append_tokens(cache1, 0, k, v, batch.qo_indptr, batch.page_table, batch.seq_lens,
                            batch.active)
    out1, lse1, _ = oracle.prefill_attn(cache1, 0, q, batch.qo_indptr, batch.page_table,
                                        batch.seq_lens, batch.active)
    cache2 = W.bf16_bits(t.cache)
    outs = []
    for lo, hi in ((0, 64), (64, 150)):
        ind = np.array([0, hi - lo], np.int32)
        sl = np.array([30 + hi], np.int32)
        oracle.kv_append_tokens(cache2, 0, k[lo:hi], v[lo:hi], ind, batch.page_table, sl,
                                batch.active)
        o, l_, _ = oracle.prefill_attn(cache2, 0, q[lo:hi], ind, batch.page_table, sl,
                                       batch.active)
        outs.append((o, l_))
    np.testing.assert_array_equal(np.concatenate([o for o, _ in outs]), out1)
    np.testing.assert_array_equal(np.concatenate([l_ for _, l_ in outs]), lse1)
    np.testing.assert_array_equal(cache2, cache1)


def test_append_tokens_bytes():
    cfg = W.PREFILL_CONFIGS["prefill_tiny"]
    batch, t = _inputs(cfg)
    before = W.bf16_bits(t.cache)
    got = before.copy()
    k, v = W.bf16_bits(t.k[0]), W.bf16_bits(t.v[0])
    assert oracle.kv_append_tokens(got, 0, k, v, batch.qo_indptr, batch.page_table,
                                   batch.seq_lens, batch.active) == 0
    want = before.copy()
    ps = cfg.page_size
    for b in range(batch.B):
        if not batch.active[b]:
            continue
        n, nq = int(batch.seq_lens[b]), batch.new_tokens(b)
        for i in range(nq):
            pos = n - nq + i
            pg = batch.page_table[b, pos // ps]
            want[0, pg, 0, pos % ps] = k[batch.qo_indptr[b] + i]
            want[0, pg, 1, pos % ps] = v[batch.qo_indptr[b] + i]
    # page 0 takes the padding tokens (in some order); every other page exact
    np.testing.assert_array_equal(got[:, 1:], want[:, 1:])
    pad_b = batch.B - 1
    assert not batch.active[pad_b]
    last = batch.qo_indptr[pad_b + 1] - 1
    np.testing.assert_array_equal(got[0, 0, 0, 0], k[last])


def test_malformed_requests_are_rejected_and_write_nothing():
    cfg = W.PrefillConfig(name="bad", index=36, num_layers=1, num_qo_heads=4, num_kv_heads=2,
                          head_dim=64, page_size=16, reqs=((0, 10), (5, 20)), bucket=False)
    batch, t = _inputs(cfg)
    batch.seq_lens[1] = 10  # fewer than its 20 new tokens
    cache = W.bf16_bits(t.cache)
    before = cache.copy()
    k, v = W.bf16_bits(t.k[0]), W.bf16_bits(t.v[0])
    assert oracle.kv_append_tokens(cache, 0, k, v, batch.qo_indptr, batch.page_table,
                                   batch.seq_lens, batch.active) == 1
    pg = batch.page_table[1, :2]
    np.testing.assert_array_equal(cache[0, pg], before[0, pg])
    out, lse, bad = oracle.prefill_attn(cache, 0, W.bf16_bits(t.q[0]), batch.qo_indptr,
                                        batch.page_table, batch.seq_lens, batch.active)
    assert bad == 1
    assert np.all(out[10:30] == 0) and np.all(np.isneginf(lse[10:30]))
    assert np.all(np.isfinite(lse[:10]))
