"""Failure detection without a GPU fault: every wait of the kernels is
bounded, and a wait that runs out sets PKV_DEV_ERR_TIMEOUT in the error word
and returns.  pkv_selftest_wait_timeout runs that same wait on an mbarrier
nothing completes; afterwards the context must still run a decode step
cleanly."""
import numpy as np
import pytest
import torch

import paged_kv_decode_pages_gb300 as pkv
from paged_kv_decode_pages_gb300 import workloads as W
from paged_kv_decode_pages_gb300.step import DecodeStep

pytestmark = pytest.mark.gpu

PKV_DEV_ERR_TIMEOUT = 0x8


def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    pkv.selftest_wait_timeout(20_000_000, err)  # 20 ms
    s1.record()
    torch.cuda.synchronize()
    assert int(err.item()) == PKV_DEV_ERR_TIMEOUT
    assert s0.elapsed_time(s1) >= 19.0  # it waited out its limit, no longer hung
    batch = W.make_batch(W.CONFIGS["tiny"])
    dev = W.Tensors(batch, device="cuda")
    step = DecodeStep(batch, dev)
    step.run()
    torch.cuda.synchronize()
    assert int(step.err.item()) == 0
    assert torch.isfinite(step.out.float()).all()
    assert np.all(step.out_tok.cpu().numpy() >= 0)
