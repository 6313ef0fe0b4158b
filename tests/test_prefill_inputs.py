"""Host-side checks of the prefill / mixed-step inputs and of the bench's
algorithmic FLOP count (no GPU): the token-bucket ladder, the packing of
requests, the page tables, and the causal key count against brute force."""
import numpy as np

import bench
from paged_kv_decode_pages_gb300 import workloads as W


def test_ladder_is_the_pages_bucket_list():
    assert W.LADDER == (32, 64, 128, 256, 512, 1024, 2048, 2176, 4096, 4352, 8192, 8704)
    assert W.ladder_bucket(1) == 32 and W.ladder_bucket(2049) == 2176
    assert W.ladder_bucket(4097) == 4352 and W.ladder_bucket(8700) == 8704
    assert W.ladder_bucket(9000) == 9000  # past the ladder: unpadded


def test_prefill_batches_pack_requests_and_pad_to_the_bucket():
    for name, cfg in W.PREFILL_CONFIGS.items():
        b = W.make_prefill_batch(cfg)
        assert b.qo_indptr[0] == 0 and np.all(np.diff(b.qo_indptr) >= 0)
        real = sum(b.new_tokens(i) for i in range(b.B) if b.active[i])
        assert b.T == W.ladder_bucket(real) if cfg.bucket else b.T == real
        ps = cfg.page_size
        used = []
        for i in range(b.B):
            if not b.active[i]:
                assert np.all(b.page_table[i] == 0)
                continue
            assert b.seq_lens[i] >= b.new_tokens(i) >= 1
            npg = (int(b.seq_lens[i]) + ps - 1) // ps
            pages = b.page_table[i, :npg]
            assert np.all(pages >= 1) and np.all(pages < b.num_pages)
            used.extend(pages.tolist())
        assert len(used) == len(set(used))  # no page shared between requests


def test_prefill_flops_count_each_tokens_causal_keys():
    cfg = W.PREFILL_CONFIGS["prefill_tiny"]
    b = W.make_prefill_batch(cfg)
    keys = 0
    for i in range(b.B):
        if not b.active[i]:
            continue
        n, q = int(b.seq_lens[i]), b.new_tokens(i)
        keys += sum(n - q + t + 1 for t in range(q))  # token t sees positions 0..n-q+t
    assert bench.prefill_flops(b) == 4.0 * cfg.head_dim * cfg.num_qo_heads * keys
