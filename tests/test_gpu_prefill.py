"""GPU parity of the prefill / mixed step (kv_append_tokens, then the tensor-
core prefill_attn) against the fp64 oracle on the same seeded inputs.

Tolerances as for decode attention (bf16 inputs, fp32 accumulation, one bf16
rounding of the output; P rounded to bf16 before P.V): max-abs 1e-2 and
mean-abs 1e-3 on the outputs, 1e-3 on lse; the append bit-exact on every
page but the dummy page 0."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_pages_gb300 import workloads as W
from paged_kv_decode_pages_gb300.step import PrefillStep

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 1e-2, 1e-3, 1e-3

CASES = {
    "tiny_g4_d64": W.PREFILL_CONFIGS["prefill_tiny"],
    "g1_d128_p32": W.PrefillConfig(name="g1", index=30, num_layers=1, num_qo_heads=3,
                                   num_kv_heads=3, head_dim=128, page_size=32,
                                   reqs=((0, 33), (40, 1), (7, 70)), shuffle_pages=True),
    "g7_d64_p128": W.PrefillConfig(name="g7", index=31, num_layers=2, num_qo_heads=14,
                                   num_kv_heads=2, head_dim=64, page_size=128,
                                   reqs=((200, 60), (0, 129), (127, 2)), bucket=False),
    "mixed_g4_d128": W.PrefillConfig(
        name="mixed_small", index=40, num_layers=2, num_qo_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, n_prefill=3, prefix_lo=0, prefix_hi=700, new_lo=100,
        new_hi=400, n_decode=9, ctx_lo=30, ctx_hi=1500),
    "p128_g4_d128": W.PrefillConfig(
        name="p128_small", index=41, num_layers=1, num_qo_heads=32, num_kv_heads=8,
        head_dim=128, page_size=128, reqs=((0, 300), (129, 257), (1000, 1), (0, 1)),
        shuffle_pages=True),
    # 33-64 requests: the unit lookup takes a second 32-position ballot
    "requests_45": W.PrefillConfig(
        name="req45", index=44, num_layers=1, num_qo_heads=16, num_kv_heads=4, head_dim=128,
        page_size=32, reqs=tuple(((11 * i) % 150, 1 + (17 * i) % 70) for i in range(45)),
        bucket=False),
    # more than 64 requests: the kernel finds a unit's request by binary search
    "many_requests_70": W.PrefillConfig(
        name="many70", index=43, num_layers=1, num_qo_heads=8, num_kv_heads=2, head_dim=64,
        page_size=16, reqs=tuple(((7 * i) % 90, 1 + (13 * i) % 40) for i in range(70)),
        bucket=False),
    "g8_d128_long_prefix": W.PrefillConfig(
        name="long_prefix", index=42, num_layers=1, num_qo_heads=16, num_kv_heads=2,
        head_dim=128, page_size=16, reqs=((3000, 40), (2047, 129), (0, 16)), bucket=False),
}


def _run(cfg):
    batch = W.make_prefill_batch(cfg)
    host = W.PrefillTensors(batch, device="cpu")
    cache_bits = W.bf16_bits(host.cache)
    dev = W.PrefillTensors.__new__(W.PrefillTensors)
    dev.cache = host.cache.cuda()
    dev.q, dev.k, dev.v = host.q.cuda(), host.k.cuda(), host.v.cuda()
    dev.layers = host.layers
    step = PrefillStep(batch, dev)
    step.run()
    torch.cuda.synchronize()
    return batch, host, cache_bits, step


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_step_matches_oracle(name):
    cfg = CASES[name]
    batch, host, cache_bits, step = _run(cfg)
    assert int(step.err.item()) == 0
    pad = np.zeros(batch.T, bool)
    for b in range(batch.B):
        if not batch.active[b]:
            pad[batch.qo_indptr[b]:batch.qo_indptr[b + 1]] = True
    worst = 0.0
    for l in range(host.layers):
        assert oracle.kv_append_tokens(cache_bits, l, W.bf16_bits(host.k[l]),
                                       W.bf16_bits(host.v[l]), batch.qo_indptr, batch.page_table,
                                       batch.seq_lens, batch.active) == 0
        want, want_lse, bad = oracle.prefill_attn(cache_bits, l, W.bf16_bits(host.q[l]),
                                                  batch.qo_indptr, batch.page_table,
                                                  batch.seq_lens, batch.active)
        assert bad == 0
        got = step.out[l].float().cpu().numpy().astype(np.float64)
        err = np.abs(got - want)
        assert err.max() <= MAX_ABS, (name, l, err.max(), np.unravel_index(err.argmax(), err.shape))
        assert err.mean() <= MEAN_ABS, (name, l, err.mean())
        worst = max(worst, float(err.max()))
        lse = step.lse[l].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(lse[~pad] - want_lse[~pad]) <= LSE_ABS), (name, l)
        assert np.all(np.isneginf(lse[pad]))
        assert np.all(got[pad] == 0.0)
    got_cache = W.bf16_bits(step.t.cache)
    np.testing.assert_array_equal(got_cache[:, 1:], cache_bits[:, 1:])
    print(name, "worst max-abs", worst)


def test_prefill_rows_do_not_depend_on_the_other_requests():
    """A request alone or inside the mixed batch: bit-identical outputs."""
    cfg = CASES["mixed_g4_d128"]
    batch, host, _, step = _run(cfg)
    b = 1
    lo, hi = int(batch.qo_indptr[b]), int(batch.qo_indptr[b + 1])
    one = W.PrefillBatch(cfg, np.array([0, hi - lo], np.int32), batch.seq_lens[b:b + 1].copy(),
                         batch.active[b:b + 1].copy(), batch.page_table[b:b + 1].copy(),
                         batch.num_pages)
    dev = W.PrefillTensors.__new__(W.PrefillTensors)
    dev.cache = host.cache.cuda()
    dev.q = host.q[:, lo:hi].contiguous().cuda()
    dev.k = host.k[:, lo:hi].contiguous().cuda()
    dev.v = host.v[:, lo:hi].contiguous().cuda()
    dev.layers = host.layers
    s1 = PrefillStep(one, dev)
    s1.run()
    torch.cuda.synchronize()
    assert torch.equal(s1.out, step.out[:, lo:hi])
    assert torch.equal(s1.lse, step.lse[:, lo:hi])


def test_stale_cache_slots_cannot_reach_the_output():
    """Slots past each request's last position hold NaN: outputs unchanged."""
    cfg = CASES["mixed_g4_d128"]
    batch, host, _, step = _run(cfg)
    ps = cfg.page_size
    poisoned = host.cache.clone()
    for b in range(batch.B):
        if not batch.active[b]:
            continue
        n = int(batch.seq_lens[b])
        last = batch.page_table[b, (n - 1) // ps]
        poisoned[:, last, :, (n - 1) % ps + 1:] = float("nan")
    dev = W.PrefillTensors.__new__(W.PrefillTensors)
    dev.cache = poisoned.cuda()
    dev.q, dev.k, dev.v = host.q.cuda(), host.k.cuda(), host.v.cuda()
    dev.layers = host.layers
    s2 = PrefillStep(batch, dev)
    s2.run()
    torch.cuda.synchronize()
    assert torch.equal(s2.out, step.out)


def test_malformed_request_is_reported_and_zeroed():
    cfg = CASES["tiny_g4_d64"]
    batch = W.make_prefill_batch(cfg)
    batch.seq_lens[2] = 10  # fewer than its 40 new tokens
    host = W.PrefillTensors(batch, device="cpu")
    dev = W.PrefillTensors.__new__(W.PrefillTensors)
    dev.cache = host.cache.cuda()
    dev.q, dev.k, dev.v = host.q.cuda(), host.k.cuda(), host.v.cuda()
    dev.layers = host.layers
    step = PrefillStep(batch, dev)
    step.run()
    torch.cuda.synchronize()
    assert int(step.err.item()) & 0x2
    lo, hi = int(batch.qo_indptr[2]), int(batch.qo_indptr[3])
    assert torch.all(step.out[:, lo:hi] == 0)
    assert torch.all(torch.isneginf(step.lse[:, lo:hi]))
