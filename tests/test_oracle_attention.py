"""Pins of the oracle's paged decode attention and KV append against things
other than itself: torch's fp64 scaled_dot_product_attention on the dense
sequence, closed forms (identical keys -> mean of V, one token -> v, all-ones
V -> ones), log-sum-exp merging of two halves, page-placement invariance and
exact bytes for the append.

Layout and semantics follow "Adding a Model" (vox-serve docs), section
"1. The model code" (cache [num_layers, num_pages, 2, page_size,
num_kv_heads, head_dim]; set_kv_cache / run) and section "How a program
runs" (padding entries point at KV page 0 and never write other requests'
state)."""
import numpy as np
import pytest
import torch

import oracle

PS = 16


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def _from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


def _random_setup(seed=0, L=2, Hkv=2, G=4, D=64, ctx=(1, 17, 64, 200), shuffle=True, n_pad=1):
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    npg = [(n + PS - 1) // PS for n in ctx]
    P = 1 + sum(npg) + 3  # a few pages nobody owns
    ids = np.arange(1, 1 + sum(npg))
    if shuffle:
        ids = rng.permutation(ids)
    B = len(ctx) + n_pad
    max_pages = max(npg) + 2
    pt = np.zeros((B, max_pages), np.int32)
    o = 0
    for b, n in enumerate(npg):
        pt[b, :n] = ids[o:o + n]
        o += n
    seq = np.ones(B, np.int32)
    seq[: len(ctx)] = ctx
    act = np.zeros(B, np.int32)
    act[: len(ctx)] = 1
    cache = torch.randn((L, P, 2, PS, Hkv, D), generator=g).to(torch.bfloat16)
    q = torch.randn((B, Hkv * G, D), generator=g).to(torch.bfloat16)
    return dict(cache=_bits(cache), q=_bits(q), pt=pt, seq=seq, act=act, L=L, Hkv=Hkv, G=G, D=D)


def _dense_kv(cache_bits, layer, pt, b, n):
    """Gather K, V of row b ([n, Hkv, D] fp64) by walking its page table."""
    c = _from_bits(cache_bits).double()
    pages = [int(pt[b, t // PS]) for t in range(n)]
    slots = [t % PS for t in range(n)]
    K = torch.stack([c[layer, p, 0, s] for p, s in zip(pages, slots)])
    V = torch.stack([c[layer, p, 1, s] for p, s in zip(pages, slots)])
    return K, V


@pytest.mark.parametrize("G,D,shuffle", [(4, 64, True), (7, 64, False), (3, 128, True), (1, 32, True)])
def test_attention_matches_torch_sdpa_fp64(G, D, shuffle):
    s = _random_setup(seed=G * 100 + D, G=G, D=D, shuffle=shuffle)
    Hq = s["Hkv"] * G
    for layer in range(s["L"]):
        out, lse, bad = oracle.paged_decode_attn(s["cache"], layer, s["q"], s["pt"], s["seq"], s["act"])
        assert bad == 0
        for b in range(len(s["seq"])):
            if not s["act"][b]:
                assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
                continue
            n = int(s["seq"][b])
            K, V = _dense_kv(s["cache"], layer, s["pt"], b, n)
            # [Hq, n, D] with kv head h // G for q head h
            Kq = K.permute(1, 0, 2).repeat_interleave(G, dim=0)
            Vq = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
            qd = _from_bits(s["q"][b]).double().unsqueeze(1)  # [Hq, 1, D]
            ref = torch.nn.functional.scaled_dot_product_attention(qd, Kq, Vq).squeeze(1)
            np.testing.assert_allclose(out[b], ref.numpy(), rtol=0, atol=1e-12)
            scores = (qd @ Kq.transpose(1, 2)).squeeze(1) / np.sqrt(D)
            ref_lse = torch.logsumexp(scores, dim=-1)
            np.testing.assert_allclose(lse[b], ref_lse.numpy(), rtol=0, atol=1e-12)
            assert out.shape == (len(s["seq"]), Hq, D)


def test_identical_keys_give_mean_of_values():
    s = _random_setup(seed=3, G=4, D=64)
    cache = s["cache"].copy()
    b = 3
    n = int(s["seq"][b])
    key_row = cache[0, int(s["pt"][b, 0]), 0, 0].copy()  # [Hkv, D]
    for t in range(n):
        cache[0, int(s["pt"][b, t // PS]), 0, t % PS] = key_row
    out, _, _ = oracle.paged_decode_attn(cache, 0, s["q"], s["pt"], s["seq"], s["act"])
    _, V = _dense_kv(cache, 0, s["pt"], b, n)
    mean_v = V.mean(dim=0).numpy()  # [Hkv, D]
    for h in range(s["Hkv"] * s["G"]):
        np.testing.assert_allclose(out[b, h], mean_v[h // s["G"]], rtol=0, atol=1e-13)


def test_single_token_returns_its_value():
    s = _random_setup(seed=5)
    out, lse, _ = oracle.paged_decode_attn(s["cache"], 1, s["q"], s["pt"], s["seq"], s["act"])
    assert s["seq"][0] == 1
    _, V = _dense_kv(s["cache"], 1, s["pt"], 0, 1)
    for h in range(s["Hkv"] * s["G"]):
        np.testing.assert_array_equal(out[0, h], V[0, h // s["G"]].numpy())


def test_all_ones_values_give_ones():
    """Softmax weights sum to one: with every V row all ones the output is
    all ones."""
    s = _random_setup(seed=7, G=4, D=64, ctx=(300, 5, 1000))
    cache = s["cache"].copy()
    cache[:, :, 1] = _bits(torch.ones(1))[0]
    out, _, _ = oracle.paged_decode_attn(cache, 0, s["q"], s["pt"], s["seq"], s["act"])
    act = s["act"].astype(bool)
    np.testing.assert_allclose(out[act], 1.0, rtol=0, atol=1e-13)


def test_page_placement_permutation_is_bit_identical():
    s = _random_setup(seed=11, ctx=(33, 200, 129), shuffle=False)
    cache = s["cache"]
    P = cache.shape[1]
    rng = np.random.default_rng(1)
    perm = np.concatenate([[0], 1 + rng.permutation(P - 1)])  # page p moves to perm[p]
    moved = np.empty_like(cache)
    moved[:, perm] = cache
    pt2 = perm[s["pt"]].astype(np.int32)
    a, la, _ = oracle.paged_decode_attn(cache, 0, s["q"], s["pt"], s["seq"], s["act"])
    b, lb, _ = oracle.paged_decode_attn(moved, 0, s["q"], pt2, s["seq"], s["act"])
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_two_halves_merge_by_lse_to_the_whole():
    s = _random_setup(seed=13, ctx=(16 * 9 + 5, 16 * 4), n_pad=0)
    whole, lw, _ = oracle.paged_decode_attn(s["cache"], 0, s["q"], s["pt"], s["seq"], s["act"])
    for b in range(2):
        n = int(s["seq"][b])
        npg = (n + PS - 1) // PS
        k = npg // 2
        pt1 = s["pt"][b:b + 1].copy()
        pt2 = np.zeros_like(pt1)
        pt2[0, : npg - k] = s["pt"][b, k:npg]
        qb = s["q"][b:b + 1]
        o1, l1, _ = oracle.paged_decode_attn(s["cache"], 0, qb, pt1, np.array([k * PS], np.int32),
                                             np.ones(1, np.int32))
        o2, l2, _ = oracle.paged_decode_attn(s["cache"], 0, qb, pt2, np.array([n - k * PS], np.int32),
                                             np.ones(1, np.int32))
        m = np.maximum(l1, l2)
        w1 = np.exp(l1 - m)[..., None]
        w2 = np.exp(l2 - m)[..., None]
        merged = (w1 * o1 + w2 * o2) / (w1 + w2)
        np.testing.assert_allclose(merged[0], whole[b], rtol=0, atol=1e-13)
        np.testing.assert_allclose((m + np.log(w1[..., 0] + w2[..., 0]))[0], lw[b], rtol=0, atol=1e-13)


def test_bad_rows_are_rejected_and_others_unaffected():
    s = _random_setup(seed=17, ctx=(40, 70))
    ref, _, _ = oracle.paged_decode_attn(s["cache"], 0, s["q"], s["pt"], s["seq"], s["act"])
    pt = s["pt"].copy()
    pt[0, 1] = 10 ** 6  # page id out of range
    seq = s["seq"].copy()
    out, _, bad = oracle.paged_decode_attn(s["cache"], 0, s["q"], pt, seq, s["act"])
    assert bad == 1 and np.all(out[0] == 0)
    np.testing.assert_array_equal(out[1], ref[1])
    seq[1] = pt.shape[1] * PS + 1  # longer than the page table
    out, _, bad = oracle.paged_decode_attn(s["cache"], 0, s["q"], pt, seq, s["act"])
    assert bad == 2 and np.all(out[1] == 0)


# ---------------------------------------------------------------------------
# KV append
# ---------------------------------------------------------------------------
def test_append_writes_exactly_the_slot_and_nothing_else():
    s = _random_setup(seed=19, ctx=(1, 17, 64, 200), n_pad=2)
    B = len(s["seq"])
    g = torch.Generator().manual_seed(2)
    k = _bits(torch.randn((B, s["Hkv"], s["D"]), generator=g))
    v = _bits(torch.randn((B, s["Hkv"], s["D"]), generator=g))
    cache = s["cache"].copy()
    before = cache.copy()
    bad = oracle.kv_append(cache, 1, k, v, s["pt"], s["seq"], s["act"])
    assert bad == 0
    expect = before.copy()
    for b in range(B):
        if s["act"][b]:
            pos = int(s["seq"][b]) - 1
            page, slot = int(s["pt"][b, pos // PS]), pos % PS
        else:
            page, slot = 0, 0
        expect[1, page, 0, slot] = k[b]
        expect[1, page, 1, slot] = v[b]
    np.testing.assert_array_equal(cache, expect)
    # layer 0 untouched; pages other than the written slots and page 0 untouched
    np.testing.assert_array_equal(cache[0], before[0])
    changed = np.argwhere(np.any(cache != before, axis=(2, 3, 4, 5)))
    owned = {(1, int(s["pt"][b, (int(s["seq"][b]) - 1) // PS])) for b in range(B) if s["act"][b]}
    for l, p in changed:
        assert (int(l), int(p)) in owned or p == 0


def test_append_rejects_out_of_range_rows():
    s = _random_setup(seed=23, ctx=(5, 9))
    B = len(s["seq"])
    k = np.full((B, s["Hkv"], s["D"]), 0x3F80, np.uint16)
    cache = s["cache"].copy()
    before = cache.copy()
    pt = s["pt"].copy()
    pt[1, 0] = -3
    seq = s["seq"].copy()
    seq[0] = 0
    bad = oracle.kv_append(cache, 0, k, k, pt, seq, s["act"])
    assert bad == 2
    diff = np.argwhere(np.any(cache != before, axis=(2, 3, 4, 5)))
    assert all(p == 0 for _, p in diff)  # only the padding row's dummy page
