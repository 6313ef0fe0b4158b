"""Full-size parity: each configuration's whole step (every layer's append and
attention, the sampler, the frame loop) runs at its full size, launched
call by call and as the one captured CUDA graph that bench.py replays (the
step's single attention plan, then every layer); the oracle then recomputes
sampled outputs one by one (two rows at the first and last layer) from the
inputs drawn before the step ran, plus every row of the sampler and the
frame.  The graph of the attention calls alone, which bench.py times for the
roofline, is checked the same way."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_pages_gb300 import workloads as W
from paged_kv_decode_pages_gb300.step import DecodeStep

pytestmark = pytest.mark.gpu

NEAR = 1e-6


def _snapshot(dev, batch, layer, b):
    """The pre-append pages of row b at `layer`, as a compact one-layer cache
    whose page 0 is a dummy, with the row's page table remapped to 1..n."""
    npg = batch.npages(b)
    pages = torch.as_tensor(batch.page_table[b, :npg].astype(np.int64), device=dev.cache.device)
    body = dev.cache[layer].index_select(0, pages)
    compact = torch.zeros((1, npg + 1) + tuple(body.shape[1:]), dtype=body.dtype)
    compact[0, 1:] = body.cpu()
    pt = np.zeros((1, npg), np.int32)
    pt[0] = np.arange(1, npg + 1)
    return W.bf16_bits(compact), pt


def _check_attention(name, cfg, batch, step, snaps, qkv):
    """The sampled (layer, row) outputs of step.out / step.lse against the
    oracle; returns the worst max-abs error."""
    worst = 0.0
    for (l, b), (cbits, pt) in snaps.items():
        q, k, v = qkv[(l, b)]
        sl = batch.seq_lens[b:b + 1]
        one = np.ones(1, np.int32)
        cb = cbits.copy()
        assert oracle.kv_append(cb, 0, k, v, pt, sl, one) == 0
        want, want_lse, bad = oracle.paged_decode_attn(cb, 0, q, pt, sl, one)
        assert bad == 0
        got = step.out[l, b].float().cpu().numpy().astype(np.float64)
        err = np.abs(got - want[0])
        assert err.max() <= 1e-2 and err.mean() <= 1e-3, (name, l, b, err.max(), err.mean())
        worst = max(worst, float(err.max()))
        lse = step.lse[l, b].cpu().numpy().astype(np.float64)
        assert np.abs(lse - want_lse[0]).max() <= 1e-3
        # the appended slot holds exactly the new k, v
        n = int(batch.seq_lens[b])
        page = int(batch.page_table[b, (n - 1) // cfg.page_size])
        slot_kv = W.bf16_bits(step.t.cache[l, page, :, (n - 1) % cfg.page_size])
        np.testing.assert_array_equal(slot_kv[0], k[0])
        np.testing.assert_array_equal(slot_kv[1], v[0])
    # padding rows: zeros
    pad = batch.active == 0
    if pad.any():
        assert torch.all(step.out[:, torch.from_numpy(pad)] == 0)
    return worst


@pytest.mark.parametrize("mode", ["eager", "graph"])
@pytest.mark.parametrize("name", ["qwen2_0p5b", "llama3_3b", "qwen3_4b_frame", "long_context",
                                  "long_context_p128"])
def test_full_size_step_sampled_rows(name, mode):
    cfg = W.CONFIGS[name]
    batch = W.make_batch(cfg)
    dev = W.Tensors(batch, device="cuda")
    L = cfg.num_layers
    rows = [0, cfg.n_active - 1]
    layers = [0, L - 1]
    snaps = {(l, b): _snapshot(dev, batch, l, b) for l in layers for b in rows}
    logits = dev.logits.cpu().numpy()
    base = None if dev.base is None else dev.base.cpu().numpy()
    fb = None if dev.fb is None else dev.fb.cpu().numpy()
    ctrl = None if dev.ctrl is None else dev.ctrl.cpu().numpy()
    qkv = {(l, b): (W.bf16_bits(dev.q[l, b:b + 1]), W.bf16_bits(dev.k[l, b:b + 1]),
                    W.bf16_bits(dev.v[l, b:b + 1])) for l in layers for b in rows}

    step = DecodeStep(batch, dev)
    if mode == "eager":
        steps0 = batch.steps.copy()
        step.run()
    else:
        # as bench.py: capture the whole step (one plan, every layer, the
        # sampler and the frame; a warm-up step runs first and advances the
        # step counters), then replay it once into cleared outputs
        step.capture()
        torch.cuda.synchronize()
        steps0 = step.steps.cpu().numpy().copy()
        step.out.fill_(float("nan"))
        step.lse.fill_(float("nan"))
        step.out_tok.fill_(-1)
        if base is not None:
            step.out_codes.fill_(-9)
        step.replay()
    torch.cuda.synchronize()
    assert int(step.err.item()) == 0

    worst = _check_attention(name, cfg, batch, step, snaps, qkv)
    if mode == "graph":
        # the attention calls alone, as timed for the roofline
        step.capture_attention()
        step.out.fill_(float("nan"))
        step.lse.fill_(float("nan"))
        step.replay_attention()
        torch.cuda.synchronize()
        assert int(step.err.item()) == 0
        worst = max(worst, _check_attention(name, cfg, batch, step, snaps, qkv))

    # sampler: every row
    s_steps = steps0.copy()
    tok, kind, info, bad = oracle.seeded_sample(logits, batch.slots, batch.active, batch.seeds,
                                                s_steps, batch.temperature, batch.top_k,
                                                batch.top_p)
    got_tok = step.out_tok.cpu().numpy()
    near = (info["top2_gap_rel"] < NEAR) | (info["member_margin"] < NEAR)
    assert not np.any((got_tok != tok) & ~near), np.nonzero(got_tok != tok)
    print(name, mode, "sampler near-ties:", int(near.sum()), "attn worst max-abs:", worst)

    if base is not None:
        f_steps = s_steps.copy()
        if ctrl is not None:  # channel 0 (stop/continue), then the codes
            codes, fkind, finfo, bad = oracle.frame_sample(
                ctrl, cfg.ctrl_stop, base, fb, batch.slots, batch.active, batch.seeds, f_steps,
                batch.temperature, batch.top_k, batch.top_p)
        else:
            codes, fkind, finfo, bad = oracle.codebook_frame_sample(
                base, fb, batch.slots, batch.active, batch.seeds, f_steps, batch.temperature,
                batch.top_k, batch.top_p)
        got = step.out_codes.cpu().numpy()
        for r in range(got.shape[0]):
            for j in range(got.shape[1]):
                if got[r, j] != codes[r, j]:
                    assert (finfo[r, j]["top2_gap_rel"] < NEAR
                            or finfo[r, j]["member_margin"] < NEAR), (r, j)
                    break
        np.testing.assert_array_equal(step.steps.cpu().numpy(), f_steps)
    else:
        np.testing.assert_array_equal(step.steps.cpu().numpy(), s_steps)


EXT_SETTINGS = dict(min_p=0.05, rep_penalty=1.2, rep_window=-1, hist_cap=256)  # as bench.py


@pytest.mark.parametrize("name", ["qwen2_0p5b", "llama3_3b", "long_context"])
def test_full_size_sampler_ext_every_row(name):
    """seeded_sample_ext at the configuration's full batch and vocabulary, with
    the settings bench.py times (min_p, penalty over a full 256-token ring,
    both log-probs): every row against the oracle."""
    cfg = W.CONFIGS[name]
    batch = W.make_batch(cfg)
    dev = W.Tensors(batch, device="cuda")
    step = DecodeStep(batch, dev)
    step.enable_ext(**EXT_SETTINGS)
    logits = dev.logits.cpu().numpy()
    hist = step.ext_history.cpu().numpy()
    hlen = step.ext_hist_len.cpu().numpy()
    steps0 = batch.steps.copy()
    step.sample_ext()
    torch.cuda.synchronize()
    assert int(step.err.item()) == 0
    S = batch.seeds.shape[0]
    s_steps = steps0.copy()
    tok, lraw, lproc, info, bad = oracle.seeded_sample_ext(
        logits, batch.slots, batch.active, batch.seeds, s_steps, batch.temperature, batch.top_k,
        batch.top_p, min_p=np.full(S, EXT_SETTINGS["min_p"], np.float32),
        rep_penalty=np.full(S, EXT_SETTINGS["rep_penalty"], np.float32),
        rep_window=np.full(S, EXT_SETTINGS["rep_window"], np.int32), history=hist,
        hist_len=hlen)
    assert bad == 0
    got = step.out_tok.cpu().numpy()
    near = (info["top2_gap_rel"] < NEAR) | (info["member_margin"] < NEAR)
    mism = got != tok
    assert not np.any(mism & ~near), np.nonzero(mism & ~near)
    same = ~mism
    for mine, want in ((step.lp_raw, lraw), (step.lp_proc, lproc)):
        g = mine.cpu().numpy().astype(np.float64)[same]
        w = want[same].astype(np.float32)
        assert np.all(np.abs(g - w) <= 1e-7 + 2 * np.spacing(np.abs(w)).astype(np.float64))
    np.testing.assert_array_equal(step.steps.cpu().numpy(), s_steps)
    np.testing.assert_array_equal(step.ext_hist_len.cpu().numpy(), hlen)
    if not np.any(mism):
        np.testing.assert_array_equal(step.ext_history.cpu().numpy(), hist)
    print(name, "ext sampler near-ties:", int(near.sum()))


@pytest.mark.parametrize("name", ["mixed_qwen3_4b", "prefill_qwen3_4b_p128"])
def test_full_size_prefill_step_sampled_windows(name):
    """A prefill / mixed step at its full size (every layer, the launch
    configuration bench.py times); the oracle then recomputes windows of
    new tokens of sampled requests at the first and last layer from the
    cache the step left (causality: a window's outputs need only the keys
    up to its last position, all in that cache)."""
    from paged_kv_decode_pages_gb300.step import PrefillStep
    cfg = W.PREFILL_CONFIGS[name]
    batch = W.make_prefill_batch(cfg)
    dev = W.PrefillTensors(batch, device="cuda")
    q_in = {l: W.bf16_bits(dev.q[l]) for l in (0, cfg.num_layers - 1)}
    kv_in = {l: (W.bf16_bits(dev.k[l]), W.bf16_bits(dev.v[l])) for l in (0, cfg.num_layers - 1)}
    step = PrefillStep(batch, dev)
    step.run()
    torch.cuda.synchronize()
    assert int(step.err.item()) == 0
    act = [b for b in range(batch.B) if batch.active[b]]
    prompts = [b for b in act if batch.new_tokens(b) > 1]
    decodes = [b for b in act if batch.new_tokens(b) == 1]
    picks = prompts[:2] + decodes[:2]
    ps = cfg.page_size
    worst = 0.0
    for l in (0, cfg.num_layers - 1):
        for b in picks:
            n, qn = int(batch.seq_lens[b]), batch.new_tokens(b)
            lo0 = int(batch.qo_indptr[b])
            # windows: the first and the last 8 new tokens (or the only one)
            wins = [(0, min(8, qn)), (max(0, qn - 8), qn)]
            npg = (n + ps - 1) // ps
            pages = torch.as_tensor(batch.page_table[b, :npg].astype(np.int64), device="cuda")
            body = step.t.cache[l].index_select(0, pages).cpu()
            compact = torch.zeros((1, npg + 1) + tuple(body.shape[1:]), dtype=body.dtype)
            compact[0, 1:] = body
            cb = W.bf16_bits(compact)
            pt = np.arange(1, npg + 1, dtype=np.int32)[None, :]
            # the appended tokens are exactly the inputs
            kk, vv = kv_in[l]
            for i in (0, qn - 1):
                pos = n - qn + i
                got_k = W.bf16_bits(step.t.cache[l, int(batch.page_table[b, pos // ps]), 0,
                                                 pos % ps])
                np.testing.assert_array_equal(got_k, kk[lo0 + i])
            for a0, a1 in wins:
                ind = np.array([0, a1 - a0], np.int32)
                sl = np.array([n - qn + a1], np.int32)
                want, want_lse, bad = oracle.prefill_attn(cb, 0, q_in[l][lo0 + a0:lo0 + a1], ind,
                                                          pt, sl, np.ones(1, np.int32))
                assert bad == 0
                got = step.out[l, lo0 + a0:lo0 + a1].float().cpu().numpy().astype(np.float64)
                err = np.abs(got - want)
                assert err.max() <= 1e-2 and err.mean() <= 1e-3, (name, l, b, a0, err.max())
                worst = max(worst, float(err.max()))
                lse = step.lse[l, lo0 + a0:lo0 + a1].cpu().numpy().astype(np.float64)
                assert np.abs(lse - want_lse).max() <= 1e-3
    print(name, "prefill windows worst max-abs", worst)
