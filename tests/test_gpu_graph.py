"""The whole decode step (every layer's append and attention, the sampler,
the frame) captured as one CUDA graph: a replay gives bit-identical outputs
to the eager step on the same inputs, and replays read the current contents
of the step's input buffers."""
import numpy as np
import pytest
import torch

from paged_kv_decode_pages_gb300 import workloads as W
from paged_kv_decode_pages_gb300.step import DecodeStep

pytestmark = pytest.mark.gpu


def _outputs(step):
    # page 0 is the dummy page every padding row writes (in any order)
    out = {"out": step.out.clone(), "lse": step.lse.clone(),
           "cache": step.t.cache[:, 1:].clone(), "tok": step.out_tok.clone(), "kind": step.out_kind.clone(),
           "steps": step.steps.clone(), "err": step.err.clone()}
    if step.t.base is not None:
        out["codes"] = step.out_codes.clone()
        out["fkind"] = step.frame_kind.clone()
    return out


def _same(a, b):
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("cfg", [
    W.small_variant(W.CONFIGS["qwen3_4b_frame"], n_active=5, ctx_hi=1500, layers=3, n_pad=1),
    W.small_variant(W.CONFIGS["long_context_p128"], n_active=3, ctx_hi=2600, layers=2, n_pad=2,
                    vocab=40000).replace(ctx_lo=700),
], ids=["frame_step", "p128_step"])
def test_graph_replay_equals_eager(cfg):
    batch = W.make_batch(cfg)
    dev = W.Tensors(batch, device="cuda")
    step = DecodeStep(batch, dev)
    steps0 = step.steps.clone()
    cache0 = dev.cache.clone()

    step.run()
    torch.cuda.synchronize()
    eager = _outputs(step)

    dev.cache.copy_(cache0)
    step.steps.copy_(steps0)
    step.capture()
    dev.cache.copy_(cache0)
    step.steps.copy_(steps0)
    step.out.zero_()
    step.out_tok.fill_(-7)
    step.replay()
    torch.cuda.synchronize()
    _same(eager, _outputs(step))

    # new inputs written into the same buffers: the replay reads them
    gen = torch.Generator(device="cuda").manual_seed(5)
    newq = torch.randn(dev.q.shape, generator=gen, device="cuda").to(dev.q.dtype)
    newlog = torch.randn(dev.logits.shape, generator=gen, device="cuda") * 3
    for mode in ("eager", "graph"):
        dev.cache.copy_(cache0)
        step.steps.copy_(steps0)
        dev.q.copy_(newq)
        dev.logits.copy_(newlog)
        if mode == "eager":
            step.run()
        else:
            step.replay()
        torch.cuda.synchronize()
        if mode == "eager":
            want = _outputs(step)
        else:
            _same(want, _outputs(step))
    assert not torch.equal(want["out"], eager["out"])
    assert int(want["err"].item()) == 0


def test_attention_only_graph_equals_eager():
    """The attention-only graph (the bench's attention timing) computes the
    same outputs as the eager attention calls."""
    cfg = W.small_variant(W.CONFIGS["qwen2_0p5b"], n_active=9, ctx_hi=1500, layers=3)
    batch = W.make_batch(cfg)
    dev = W.Tensors(batch, device="cuda")
    step = DecodeStep(batch, dev)
    step.run()
    torch.cuda.synchronize()
    want_out, want_lse = step.out.clone(), step.lse.clone()
    step.capture_attention()
    step.out.zero_()
    step.lse.zero_()
    step.replay_attention()
    torch.cuda.synchronize()
    assert torch.equal(step.out, want_out)
    assert torch.equal(step.lse, want_lse)
    assert int(step.err.item()) == 0


def test_graph_replans_when_lengths_change():
    """The captured step holds its attention plan: a replay after the
    lengths change (every active row 517 tokens shorter, so rows cross a
    512-token split boundary) plans again and equals the eager step on the
    new lengths."""
    cfg = W.small_variant(W.CONFIGS["qwen2_0p5b"], n_active=9, ctx_hi=1500, layers=2)
    batch = W.make_batch(cfg)
    dev = W.Tensors(batch, device="cuda")
    step = DecodeStep(batch, dev)
    cache0 = dev.cache.clone()
    steps0 = step.steps.clone()
    step.capture()
    first = None
    new_lens = torch.where(step.active.bool(), torch.clamp(step.seq_lens - 517, min=1),
                           step.seq_lens)
    assert not torch.equal(new_lens, step.seq_lens)
    for mode in ("before", "eager", "graph"):
        dev.cache.copy_(cache0)
        step.steps.copy_(steps0)
        step.out.zero_()
        if mode != "before":
            step.seq_lens.copy_(new_lens)
        if mode == "graph":
            step.replay()
        else:
            step.run()
        torch.cuda.synchronize()
        if mode == "before":
            first = _outputs(step)
        elif mode == "eager":
            want = _outputs(step)
        else:
            _same(want, _outputs(step))
    assert not torch.equal(want["out"], first["out"])
    assert int(want["err"].item()) == 0
