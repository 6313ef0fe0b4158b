"""GPU parity of seeded_sample and codebook_frame_sample against the fp64
oracle on the same seeded logits: tokens bit-exact except at reported
near-ties (top two perturbed scores within 1e-6 relative, or a top-p prefix
sum within 1e-6 of p * Z), bit-identical across batch sizes and positions,
correct kinds, step counters and padding behaviour."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_pages_gb300 as pkv
from paged_kv_decode_pages_gb300 import workloads as W

pytestmark = pytest.mark.gpu

NEAR = 1e-6


class Rows:
    """Per-slot sampler state for B rows, row b on slot b + 1 (slot 0 = dummy)."""

    def __init__(self, B, temperature, top_k, top_p, seed0=0, active=None, steps0=0):
        self.B = B
        self.num_slots = B + 1
        self.slots = np.arange(1, B + 1, dtype=np.int32)
        self.active = np.ones(B, np.int32) if active is None else np.asarray(active, np.int32)
        self.slots[self.active == 0] = 0
        self.seeds = (np.arange(self.num_slots, dtype=np.uint64) * 7919 + seed0).astype(np.uint64)
        self.steps = (np.arange(self.num_slots, dtype=np.int64) * 3 + steps0).astype(np.int64)
        self.temperature = np.broadcast_to(np.float32(temperature), (self.num_slots,)).astype(np.float32).copy()
        self.top_k = np.broadcast_to(np.int32(top_k), (self.num_slots,)).astype(np.int32).copy()
        self.top_p = np.broadcast_to(np.float32(top_p), (self.num_slots,)).astype(np.float32).copy()

    def dev(self):
        d = {}
        d["slots"] = torch.from_numpy(self.slots).cuda()
        d["active"] = torch.from_numpy(self.active).cuda()
        d["seeds"] = torch.from_numpy(self.seeds.view(np.int64)).view(torch.uint64).cuda()
        d["steps"] = torch.from_numpy(self.steps.copy()).cuda()
        d["temperature"] = torch.from_numpy(self.temperature).cuda()
        d["top_k"] = torch.from_numpy(self.top_k).cuda()
        d["top_p"] = torch.from_numpy(self.top_p).cuda()
        return d


def gpu_sample(logits, rows, salt=0, advance=True, stop_tokens=None, audio_lo=0, audio_hi=0):
    x = torch.as_tensor(logits).cuda()
    B, V = x.shape
    d = rows.dev()
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    kind = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.sample_workspace_bytes(B, V), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = None if stop_tokens is None else torch.as_tensor(np.asarray(stop_tokens, np.int32)).cuda()
    pkv.seeded_sample(x, d["slots"], d["active"], d["seeds"], d["steps"], d["temperature"],
                      d["top_k"], d["top_p"], tok, kind, ws, salt=salt, advance=advance,
                      stop_tokens=st, audio_lo=audio_lo, audio_hi=audio_hi, err_word=err)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), kind.cpu().numpy(), d["steps"].cpu().numpy(), int(err.item())


def oracle_sample(logits, rows, salt=0, advance=True, stop_tokens=(), audio_lo=0, audio_hi=0):
    steps = rows.steps.copy()
    tok, kind, info, bad = oracle.seeded_sample(
        np.asarray(logits, np.float32), rows.slots, rows.active, rows.seeds, steps,
        rows.temperature, rows.top_k, rows.top_p, salt=salt, advance=advance,
        stop_tokens=stop_tokens, audio_lo=audio_lo, audio_hi=audio_hi)
    return tok, kind, steps, info


def compare(got, want, info, tag=""):
    """Bit-exact except near-ties; returns the number of near-tie rows."""
    near = (info["top2_gap_rel"] < NEAR) | (info["member_margin"] < NEAR)
    mism = got != want
    assert not np.any(mism & ~near), (tag, np.nonzero(mism & ~near), got[mism], want[mism])
    return int(np.sum(near))


def _logits(B, V, std, seed, dist="normal"):
    rng = np.random.default_rng(seed)
    if dist == "normal":
        return rng.normal(0, std, (B, V)).astype(np.float32)
    if dist == "ties":
        return rng.integers(-4, 4, (B, V)).astype(np.float32)
    if dist == "conc":  # the largest logits all in the first 8192-token chunk
        x = rng.normal(0, std, (B, V)).astype(np.float32)
        x[:, :8192] += np.float32(6.0)
        return x
    raise ValueError(dist)


# the samplers of the five configurations, at small batch
CFG_CASES = [("tiny", 5), ("qwen2_0p5b", 16), ("llama3_3b", 6), ("qwen3_4b_frame", 8),
             ("long_context", 6)]


@pytest.mark.parametrize("name,B", CFG_CASES)
def test_config_samplers_match_oracle(name, B):
    cfg = W.CONFIGS[name]
    rows = Rows(B, cfg.temperature, cfg.top_k, cfg.top_p, seed0=cfg.index,
                active=[1] * (B - 1) + [0])
    x = _logits(B, cfg.vocab, cfg.logit_std, 100 + cfg.index)
    for salt in (0, 5):
        got, gk, gsteps, err = gpu_sample(x, rows, salt=salt, stop_tokens=[3, 7], audio_lo=10,
                                          audio_hi=900)
        want, wk, wsteps, info = oracle_sample(x, rows, salt=salt, stop_tokens=[3, 7],
                                               audio_lo=10, audio_hi=900)
        assert err == 0
        n_near = compare(got, want, info, name)
        if n_near:
            print("near-ties:", name, n_near)
        agree = got == want
        np.testing.assert_array_equal(gk[agree], wk[agree])
        np.testing.assert_array_equal(gsteps, wsteps)
        assert got[-1] == 0 and gk[-1] == pkv.KIND_OTHER


@pytest.mark.parametrize("case", [
    dict(V=1024, T=0.0, k=0, p=1.0, std=2.0),          # greedy
    dict(V=1024, T=1e-6, k=5, p=0.5, std=2.0, dist="ties"),  # greedy with ties
    dict(V=3000, T=0.7, k=1, p=0.9, std=2.0, dist="ties"),   # top-k 1 with ties
    dict(V=5, T=1.0, k=0, p=0.9, std=1.0),             # vocab below the candidate count
    dict(V=20000, T=1.0, k=64, p=1.0, std=1.0),        # top-k from the chunk candidates
    dict(V=20000, T=1.0, k=65, p=0.97, std=1.0),
    dict(V=40000, T=1.0, k=256, p=0.99, std=1.0),
    dict(V=40000, T=1.0, k=512, p=0.99, std=1.0),      # top-k at the candidate count
    dict(V=40000, T=1.0, k=513, p=1.0, std=1.0),       # general path: top-k > 512
    dict(V=20000, T=2.0, k=1000, p=0.9, std=1.0),      # general path with top-p
    dict(V=20000, T=1.0, k=0, p=1.0, std=1.0),         # keep everything
    dict(V=20000, T=5.0, k=0, p=0.95, std=1.0),        # top-p needs thousands of tokens
    dict(V=20000, T=0.5, k=0, p=0.3, std=1.0),         # top-p inside the candidates
    dict(V=8193, T=0.9, k=30, p=0.8, std=3.0),         # ragged second chunk of one token
    dict(V=16384, T=1.0, k=50, p=0.9, std=1.0, dist="ties"),  # many exact ties
    dict(V=70000, T=3.0, k=0, p=0.999, std=1.0),       # general path, many blocks
    dict(V=40000, T=1.0, k=200, p=0.99, std=1.0),      # top-k above the per-chunk candidates
    dict(V=40000, T=1.0, k=300, p=0.99, std=1.0, dist="conc"),  # one chunk holds the top-k
    dict(V=151936, T=0.5, k=0, p=0.95, std=1.0, dist="conc"),   # one chunk holds the top-p set
    # the finish's bitonic union at its boundaries: 16 lists of 32 slots
    # fill 512 entries (two a thread), 17 lists take 1 024 (four a thread)
    dict(V=131072, T=0.8, k=0, p=0.9, std=2.0),
    dict(V=139264, T=0.8, k=0, p=0.9, std=2.0),
])
def test_sampler_modes_and_edges(case):
    B = 7
    rows = Rows(B, case["T"], case["k"], case["p"], seed0=case["V"])
    x = _logits(B, case["V"], case["std"], case["V"] + case["k"], case.get("dist", "normal"))
    x[2, 5 % case["V"]] = -np.inf  # masked token
    got, _, _, err = gpu_sample(x, rows)
    want, _, _, info = oracle_sample(x, rows)
    assert err == 0
    compare(got, want, info, str(case))


def test_batch_size_and_position_invariance():
    cfg = W.CONFIGS["llama3_3b"]
    V = cfg.vocab
    rng = np.random.default_rng(5)
    row = rng.normal(0, cfg.logit_std, V).astype(np.float32)
    results = []
    for B, pos in ((1, 0), (5, 4), (64, 17), (128, 127), (128, 0)):
        x = rng.normal(0, cfg.logit_std, (B, V)).astype(np.float32)
        x[pos] = row
        rows = Rows(B, cfg.temperature, cfg.top_k, cfg.top_p)
        # the row under test always sits on slot 1 with the same seed and step
        rows.slots[:] = np.arange(2, B + 2)
        rows.slots[pos] = 1
        rows.num_slots = B + 2
        rows.seeds = np.arange(B + 2, dtype=np.uint64) + 1000
        rows.steps = np.full(B + 2, 9, np.int64)
        for a in ("temperature", "top_k", "top_p"):
            setattr(rows, a, np.resize(getattr(rows, a), B + 2))
        tok, _, _, _ = gpu_sample(x, rows, salt=3)
        results.append(int(tok[pos]))
    assert len(set(results)) == 1, results
    # duplicate rows in one batch with the same slot state agree
    x = np.stack([row] * 4)
    rows = Rows(4, 0.6, 50, 0.95)
    rows.seeds[:] = 42
    rows.steps[:] = 3
    tok, _, _, _ = gpu_sample(x, rows, advance=False)
    assert len(set(tok.tolist())) == 1


def test_slot_out_of_range_is_reported_and_harmless():
    rows = Rows(3, 0.8, 20, 0.9)
    rows.slots[1] = 99
    x = _logits(3, 1024, 2.0, 1)
    got, kind, steps, err = gpu_sample(x, rows)
    assert err & 0x4
    assert got[1] == 0 and kind[1] == pkv.KIND_OTHER
    want, _, wsteps, info = oracle_sample(x, rows)
    compare(got[[0, 2]], want[[0, 2]], info[[0, 2]])
    np.testing.assert_array_equal(steps, wsteps)


def _frame(cfg, B, with_fb=True):
    from paged_kv_decode_pages_gb300.step import DecodeStep
    batch = W.make_batch(cfg.replace(n_active=B - 1, n_pad=1, num_layers=1, ctx_lo=16,
                                     ctx_hi=40))
    host = W.Tensors(batch, device="cpu", with_logits=False, with_frame=True)
    if not with_fb:
        host.fb = None
    return batch, host


def _gpu_frame(batch, host):
    d = {}
    d["slots"] = torch.from_numpy(batch.slots).cuda()
    d["active"] = torch.from_numpy(batch.active).cuda()
    d["seeds"] = torch.from_numpy(batch.seeds.view(np.int64)).view(torch.uint64).cuda()
    d["steps"] = torch.from_numpy(batch.steps.copy()).cuda()
    d["temperature"] = torch.from_numpy(batch.temperature).cuda()
    d["top_k"] = torch.from_numpy(batch.top_k).cuda()
    d["top_p"] = torch.from_numpy(batch.top_p).cuda()
    n_cb, B, V = host.base.shape
    codes = torch.empty((B, n_cb), dtype=torch.int32, device="cuda")
    kind = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.frame_workspace_bytes(n_cb, B, V), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.codebook_frame_sample(host.base.cuda(), None if host.fb is None else host.fb.cuda(),
                              d["slots"], d["active"], d["seeds"], d["steps"], d["temperature"],
                              d["top_k"], d["top_p"], codes, kind, ws, err_word=err)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), kind.cpu().numpy(), d["steps"].cpu().numpy(), int(err.item())


@pytest.mark.parametrize("with_fb", [True, False])
def test_frame_matches_oracle_full_size(with_fb):
    cfg = W.CONFIGS["qwen3_4b_frame"]
    batch, host = _frame(cfg, 33, with_fb)  # the 32 rows of the configuration + 1 padding row
    codes, kind, steps, err = _gpu_frame(batch, host)
    assert err == 0
    wsteps = batch.steps.copy()
    wcodes, wkind, info, bad = oracle.codebook_frame_sample(
        host.base.numpy(), None if host.fb is None else host.fb.numpy(), batch.slots,
        batch.active, batch.seeds, wsteps, batch.temperature, batch.top_k, batch.top_p)
    assert bad == 0
    np.testing.assert_array_equal(kind, wkind)
    np.testing.assert_array_equal(steps, wsteps)
    # row by row: identical up to the first near-tie, after which the feedback
    # may legitimately diverge
    for b in range(codes.shape[0]):
        for j in range(codes.shape[1]):
            if codes[b, j] != wcodes[b, j]:
                nt = info[b, j]
                assert nt["top2_gap_rel"] < NEAR or nt["member_margin"] < NEAR, (b, j)
                break


def test_frame_without_feedback_equals_salted_samples():
    cfg = W.CONFIGS["qwen3_4b_frame"]
    batch, host = _frame(cfg, 9, with_fb=False)
    codes, _, _, _ = _gpu_frame(batch, host)
    rows = Rows(9, cfg.temperature, cfg.top_k, cfg.top_p)
    rows.slots, rows.active = batch.slots.copy(), batch.active.copy()
    rows.num_slots = batch.num_slots
    rows.seeds, rows.steps = batch.seeds.copy(), batch.steps.copy()
    rows.temperature, rows.top_k, rows.top_p = batch.temperature, batch.top_k, batch.top_p
    for j in range(cfg.n_codebooks):
        tok, _, _, _ = gpu_sample(host.base[j].numpy(), rows, salt=1 + j, advance=False)
        np.testing.assert_array_equal(codes[:, j][batch.active == 1], tok[batch.active == 1])


# ---------------------------------------------------------------------------
# Full frame: stop/continue on channel 0 gating the codebooks
# ---------------------------------------------------------------------------
def _gpu_full_frame(batch, host, ctrl, stop):
    d = {}
    d["slots"] = torch.from_numpy(batch.slots).cuda()
    d["active"] = torch.from_numpy(batch.active).cuda()
    d["seeds"] = torch.from_numpy(batch.seeds.view(np.int64)).view(torch.uint64).cuda()
    d["steps"] = torch.from_numpy(batch.steps.copy()).cuda()
    d["temperature"] = torch.from_numpy(batch.temperature).cuda()
    d["top_k"] = torch.from_numpy(batch.top_k).cuda()
    d["top_p"] = torch.from_numpy(batch.top_p).cuda()
    n_cb, B, V = host.base.shape
    rows = torch.full((B, 1 + n_cb), -7, dtype=torch.int32, device="cuda")
    kind = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.frame_sample_workspace_bytes(n_cb, B, V, ctrl.shape[1]),
                     dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.frame_sample(torch.from_numpy(ctrl).cuda(), stop, host.base.cuda(),
                     None if host.fb is None else host.fb.cuda(), d["slots"], d["active"],
                     d["seeds"], d["steps"], d["temperature"], d["top_k"], d["top_p"], rows, kind,
                     ws, err_word=err)
    torch.cuda.synchronize()
    return rows.cpu().numpy(), kind.cpu().numpy(), d["steps"].cpu().numpy(), int(err.item())


def _compare_frame_rows(got, want, info):
    """Identical up to the first near-tie of a row, after which the feedback
    may legitimately diverge."""
    for b in range(got.shape[0]):
        for j in range(got.shape[1]):
            if got[b, j] != want[b, j]:
                nt = info[b, j]
                assert nt["top2_gap_rel"] < NEAR or nt["member_margin"] < NEAR, (b, j)
                break


@pytest.mark.parametrize("ctrl_vocab,stop,bias", [
    (2, 1, -1.0),      # the configuration's channel 0: continue / stop
    (2, 1, 0.0),       # about half the rows stop
    (300, 17, 2.0),    # a larger control vocabulary (a single chunk)
    (9000, 8191, 4.0), # control vocabulary over two chunks, stop in the first
])
def test_full_frame_matches_oracle(ctrl_vocab, stop, bias):
    cfg = W.CONFIGS["qwen3_4b_frame"]
    batch, host = _frame(cfg, 33, True)  # the 32 rows of the configuration + 1 padding row
    rng = np.random.default_rng(ctrl_vocab + stop)
    ctrl = rng.normal(0, 1.0, (batch.B, ctrl_vocab)).astype(np.float32)
    ctrl[:, stop] += np.float32(bias)
    rows, kind, steps, err = _gpu_full_frame(batch, host, ctrl, stop)
    assert err == 0
    wsteps = batch.steps.copy()
    wrows, wkind, info, bad = oracle.frame_sample(ctrl, stop, host.base.numpy(), host.fb.numpy(),
                                                  batch.slots, batch.active, batch.seeds, wsteps,
                                                  batch.temperature, batch.top_k, batch.top_p)
    assert bad == 0
    np.testing.assert_array_equal(steps, wsteps)
    _compare_frame_rows(rows, wrows, info)
    agree = rows[:, 0] == wrows[:, 0]
    np.testing.assert_array_equal(kind[agree], wkind[agree])
    stopped = (rows[:, 0] == stop) & (batch.active == 1)
    assert np.all(rows[stopped, 1:] == pkv.CODE_PAD)
    assert np.all(kind[stopped] == pkv.KIND_STOP)
    assert np.all(kind[(rows[:, 0] != stop) & (batch.active == 1)] == pkv.KIND_AUDIO)
    assert np.all(rows[batch.active == 0] == 0)


def test_full_frame_stop_and_continue_both_occur_in_the_configuration():
    cfg = W.CONFIGS["qwen3_4b_frame"]
    batch = W.make_batch(cfg)
    host = W.Tensors(batch, device="cpu", layers=1, with_logits=False, with_frame=True)
    rows, kind, _, err = _gpu_full_frame(batch, host, host.ctrl.numpy(), cfg.ctrl_stop)
    assert err == 0
    act = batch.active == 1
    n_stop = int((kind[act] == pkv.KIND_STOP).sum())
    assert 0 < n_stop < int(act.sum()), n_stop


def test_full_frame_rejects_a_stop_token_outside_the_control_vocabulary():
    cfg = W.CONFIGS["qwen3_4b_frame"]
    batch, host = _frame(cfg, 5, True)
    ctrl = np.zeros((batch.B, 2), np.float32)
    with pytest.raises(pkv.PkvError) as e:
        _gpu_full_frame(batch, host, ctrl, 2)
    assert e.value.status == 1  # PKV_ERR_INVALID_ARG
