"""GPU parity of seeded_sample_ext (repetition penalty over a per-slot token
history, temperature, top-k, min_p, top-p; raw and processed log-probs)
against the fp64 oracle on the same seeded inputs: tokens bit-exact except
at reported near-ties, log-probs within two fp32 ulps (+1e-7) of the
oracle's fp32 values, history rings, history lengths and step counters
exact, and rows independent of the batch they are sampled in."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_pages_gb300 as pkv

pytestmark = pytest.mark.gpu

NEAR = 1e-6
CAP = 32


def _lp_close(got, want):
    want = np.asarray(want, np.float32)
    return (np.abs(got.astype(np.float64) - want.astype(np.float64))
            <= 1e-7 + 2 * np.spacing(np.abs(want)).astype(np.float64))


class ExtRows:
    """B rows, row b on slot b + 1 (slot 0 = dummy), with per-slot settings
    cycled from the given lists and a wrapped history ring that holds each
    row's own leading tokens (so the penalty changes the order)."""

    def __init__(self, x, T, k, p, min_p, pen, window, seed0=0, active=None, hist_len0=40):
        B, V = x.shape
        self.B, self.V = B, V
        S = B + 1
        self.num_slots = S
        self.active = np.ones(B, np.int32) if active is None else np.asarray(active, np.int32)
        self.slots = np.arange(1, B + 1, dtype=np.int32)
        self.slots[self.active == 0] = 0
        cyc = lambda v, dt: np.resize(np.asarray(v, dt), S).astype(dt)  # noqa: E731
        self.seeds = (np.arange(S, dtype=np.uint64) * 104729 + seed0).astype(np.uint64)
        self.steps = (np.arange(S, dtype=np.int64) * 5 + 11).astype(np.int64)
        self.temperature = cyc(T, np.float32)
        self.top_k = cyc(k, np.int32)
        self.top_p = cyc(p, np.float32)
        self.min_p = cyc(min_p, np.float32)
        self.pen = cyc(pen, np.float32)
        self.window = cyc(window, np.int32)
        rng = np.random.default_rng(seed0 + 17)
        self.history = rng.integers(0, V, (S, CAP)).astype(np.int32)
        self.hist_len = np.full(S, hist_len0, np.int32)
        self.hist_len[::3] = 5  # some rings not yet full
        for b in range(B):
            s = self.slots[b]
            if s == 0:
                continue
            lead = np.argsort(-x[b], kind="stable")[:5].astype(np.int32)
            n = int(self.hist_len[s])
            for i, t in enumerate(list(lead) + [lead[0]]):
                if 3 * i < min(n, CAP):
                    self.history[s, (n - 1 - 3 * i) % CAP] = t

    def dev(self):
        c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        return dict(slots=c(self.slots), active=c(self.active),
                    seeds=c(self.seeds.view(np.int64)).view(torch.uint64), steps=c(self.steps),
                    temperature=c(self.temperature), top_k=c(self.top_k), top_p=c(self.top_p),
                    min_p=c(self.min_p), rep_penalty=c(self.pen), rep_window=c(self.window),
                    history=c(self.history), hist_len=c(self.hist_len))


def gpu_ext(x, d, advance=True, want_lp=True, use=("min_p", "rep_penalty", "rep_window",
                                                    "history"), ws_bytes=None):
    xt = torch.as_tensor(x).cuda()
    B, V = xt.shape
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    kind = torch.empty(B, dtype=torch.int32, device="cuda")
    lraw = torch.full((B,), 7.0, dtype=torch.float32, device="cuda") if want_lp else None
    lproc = torch.full((B,), 7.0, dtype=torch.float32, device="cuda") if want_lp else None
    nb = pkv.sample_ext_workspace_bytes(B, V) if ws_bytes is None else ws_bytes
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.seeded_sample_ext(
        xt, d["slots"], d["active"], d["seeds"], d["steps"], d["temperature"], d["top_k"],
        d["top_p"], tok, kind, ws, min_p=d["min_p"] if "min_p" in use else None,
        rep_penalty=d["rep_penalty"] if "rep_penalty" in use else None,
        rep_window=d["rep_window"] if "rep_window" in use else None,
        history=d["history"] if "history" in use else None,
        hist_len=d["hist_len"] if "history" in use else None,
        logprob_raw=lraw, logprob_proc=lproc, advance=advance, err_word=err)
    torch.cuda.synchronize()
    out = dict(tok=tok.cpu().numpy(), kind=kind.cpu().numpy(), err=int(err.item()))
    if want_lp:
        out["lraw"] = lraw.cpu().numpy()
        out["lproc"] = lproc.cpu().numpy()
    return out


def oracle_ext(x, r, steps=None, history=None, hist_len=None, advance=True):
    steps = r.steps.copy() if steps is None else steps
    history = r.history.copy() if history is None else history
    hist_len = r.hist_len.copy() if hist_len is None else hist_len
    tok, lraw, lproc, info, bad = oracle.seeded_sample_ext(
        np.asarray(x, np.float32), r.slots, r.active, r.seeds, steps, r.temperature, r.top_k,
        r.top_p, min_p=r.min_p, rep_penalty=r.pen, rep_window=r.window, history=history,
        hist_len=hist_len, advance=advance)
    return dict(tok=tok, lraw=lraw, lproc=lproc, info=info, steps=steps, history=history,
                hist_len=hist_len)


def _check(got, want, tag=""):
    info = want["info"]
    near = (info["top2_gap_rel"] < NEAR) | (info["member_margin"] < NEAR)
    mism = got["tok"] != want["tok"]
    assert not np.any(mism & ~near), (tag, np.nonzero(mism & ~near), got["tok"], want["tok"])
    same = ~mism
    assert np.all(_lp_close(got["lraw"][same], want["lraw"][same])), (tag, got["lraw"], want["lraw"])
    assert np.all(_lp_close(got["lproc"][same], want["lproc"][same])), (tag, got["lproc"],
                                                                       want["lproc"])
    return mism


def _logits(B, V, std, seed, conc=False):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, std, (B, V)).astype(np.float32)
    if conc:
        x[:, :8192] += np.float32(6.0)
    return x


CASES = [
    # name, B, V, std, T list, k list, p list, min_p list, penalty list, window list
    ("tts-small", 16, 6561, 3.0, [1.0, 0.8], [25, 0], [0.8, 1.0], [0.0, 0.05, 0.2],
     [1.0, 1.3, 2.0], [-1, 8]),
    ("qwen-vocab", 12, 151936, 4.0, [0.7, 1.0], [0, 50], [0.95, 1.0], [0.0, 0.01],
     [1.1, 1.0, 1.5], [-1, 4, 0]),
    ("llama-vocab", 8, 128256, 4.0, [0.6], [50, 0], [0.95], [0.0, 0.1], [1.2], [-1]),
    ("greedy-pen", 8, 20000, 2.0, [0.0], [0], [1.0], [0.0], [1.0, 3.0], [-1]),
    ("keep-all", 8, 40000, 1.0, [1.0], [0], [1.0], [0.0], [1.0, 1.2], [-1]),
    ("minp-general", 6, 40000, 1.0, [1.0], [0, 700], [1.0, 0.9], [0.05, 1e-4], [1.0, 1.4], [-1]),
]


@pytest.mark.parametrize("name,B,V,std,T,k,p,mp,pen,win", CASES)
def test_ext_matches_oracle(name, B, V, std, T, k, p, mp, pen, win):
    x = _logits(B, V, std, V + B, conc=(name == "qwen-vocab"))
    x[0, 5] = -np.inf
    active = [1] * (B - 1) + [0]
    r = ExtRows(x, T, k, p, mp, pen, win, seed0=B, active=active)
    d = r.dev()
    got = gpu_ext(x, d)
    want = oracle_ext(x, r)
    assert got["err"] & ~0x10 == 0
    mism = _check(got, want, name)
    np.testing.assert_array_equal(d["steps"].cpu().numpy(), want["steps"])
    np.testing.assert_array_equal(d["hist_len"].cpu().numpy(), want["hist_len"])
    gh = d["history"].cpu().numpy()
    for b in np.nonzero(~mism)[0]:
        s = r.slots[b]
        np.testing.assert_array_equal(gh[s], want["history"][s])
    assert got["tok"][-1] == 0 and got["lraw"][-1] == 0 and got["lproc"][-1] == 0
    assert got["kind"][-1] == pkv.KIND_OTHER


def test_ext_penalty_changes_tokens_in_the_cases():
    """The cases above do exercise the penalty: switching it off changes some
    greedy tokens (oracle only, as a check of the test inputs)."""
    x = _logits(8, 20000, 2.0, 20008)
    r = ExtRows(x, [0.0], [0], [1.0], [0.0], [3.0], [-1], seed0=8)
    a = oracle_ext(x, r)["tok"]
    r.pen[:] = 1.0
    b = oracle_ext(x, r)["tok"]
    assert np.any(a != b)


def test_ext_all_off_equals_seeded_sample():
    B, V = 10, 151936
    x = _logits(B, V, 4.0, 3)
    r = ExtRows(x, [0.7, 0.0, 1.0], [0, 50, 600], [0.95, 1.0], [0.0], [1.0], [-1], seed0=3)
    d = r.dev()
    got = gpu_ext(x, d, advance=False, want_lp=False, use=())
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    kind = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.sample_workspace_bytes(B, V), dtype=torch.uint8, device="cuda")
    pkv.seeded_sample(torch.as_tensor(x).cuda(), d["slots"], d["active"], d["seeds"], d["steps"],
                      d["temperature"], d["top_k"], d["top_p"], tok, kind, ws, advance=False)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got["tok"], tok.cpu().numpy())
    np.testing.assert_array_equal(got["kind"], kind.cpu().numpy())


def test_ext_history_over_several_steps():
    """Eight steps with advance: the sampled tokens enter the ring and
    penalise the next steps exactly as in the oracle."""
    B, V = 6, 6561
    r = None
    gh = None
    for step in range(8):
        x = _logits(B, V, 3.0, 500 + step)
        if r is None:
            r = ExtRows(x, [1.0, 0.0], [25, 0], [0.8], [0.0, 0.1], [1.5, 2.5], [-1, 3], seed0=1,
                        hist_len0=0)
            r.hist_len[:] = 0
            d = r.dev()
            o_steps, o_hist, o_len = r.steps.copy(), r.history.copy(), r.hist_len.copy()
        got = gpu_ext(x, d)
        want = oracle_ext(x, r, steps=o_steps, history=o_hist, hist_len=o_len)
        mism = _check(got, want, "step %d" % step)
        if np.any(mism):  # a near-tie went the other way: the states part here
            break
        np.testing.assert_array_equal(d["history"].cpu().numpy(), o_hist)
        np.testing.assert_array_equal(d["hist_len"].cpu().numpy(), o_len)
        np.testing.assert_array_equal(d["steps"].cpu().numpy(), o_steps)
    assert int(o_len[1]) == step + 1


def test_ext_batch_size_and_position_invariance():
    B, V = 12, 151936
    x = _logits(B, V, 4.0, 77)
    r = ExtRows(x, [0.7], [0], [0.95], [0.0, 0.02], [1.0, 1.3], [-1, 6], seed0=5)
    full = gpu_ext(x, r.dev(), advance=False)
    for b in (0, 5, 11):
        sub = ExtRows(x[b:b + 1], [0.7], [0], [0.95], [0.0], [1.0], [-1], seed0=5)
        s = r.slots[b]
        for name in ("seeds", "steps", "temperature", "top_k", "top_p", "min_p", "pen", "window",
                     "hist_len"):
            getattr(sub, name)[1] = getattr(r, name)[s]
        sub.history[1] = r.history[s]
        one = gpu_ext(x[b:b + 1], sub.dev(), advance=False)
        assert one["tok"][0] == full["tok"][b]
        assert one["lraw"][0] == full["lraw"][b] and one["lproc"][0] == full["lproc"][b]


def test_ext_negative_history_length_is_reported():
    B, V = 4, 6561
    x = _logits(B, V, 3.0, 9)
    r = ExtRows(x, [1.0], [25], [0.8], [0.0], [2.0], [-1], seed0=2)
    r.hist_len[2] = -3
    d = r.dev()
    got = gpu_ext(x, d, advance=True)
    assert got["err"] & 0x20
    # that row is sampled without penalty and stores nothing
    want = oracle_ext(x, r, advance=False)
    row = 1  # slot 2
    assert got["tok"][row] == want["tok"][row] or want["info"]["member_margin"][row] < NEAR
    assert int(d["hist_len"].cpu()[2]) == -3
    np.testing.assert_array_equal(d["history"].cpu().numpy()[2], r.history[2])


def test_ext_host_argument_errors():
    B, V = 4, 6561
    x = _logits(B, V, 3.0, 9)
    r = ExtRows(x, [1.0], [25], [0.8], [0.0], [2.0], [-1], seed0=2)
    d = r.dev()
    # a penalty needs the bitmap workspace
    with pytest.raises(pkv.PkvError) as e:
        gpu_ext(x, d, ws_bytes=pkv.sample_workspace_bytes(B, V))
    assert e.value.status == 4
    # without a penalty the plain workspace suffices
    gpu_ext(x, d, use=("min_p",), ws_bytes=pkv.sample_workspace_bytes(B, V))
    # a ring of capacity 0: refused by the binding, and by the library itself
    empty = dict(d, history=torch.zeros((B + 1, 0), dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError):
        gpu_ext(x, empty)
    import ctypes
    from paged_kv_decode_pages_gb300 import _binding as Bd
    xt = torch.as_tensor(x).cuda()
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.sample_ext_workspace_bytes(B, V), dtype=torch.uint8, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    for cap, hl in ((0, d["hist_len"]), (CAP, None)):
        ext = Bd.pkv_sample_ext_t(None, p(d["rep_penalty"]), None, p(d["history"]),
                                  None if hl is None else p(hl), cap, None, None)
        st = Bd.load().pkv_seeded_sample_ext(
            p(xt), V, B, V, p(d["slots"]), p(d["active"]), B + 1, p(d["seeds"]), p(d["steps"]),
            p(d["temperature"]), p(d["top_k"]), p(d["top_p"]), 0, 1, None, 0, 0, 0, p(out),
            p(out), ctypes.byref(ext), p(ws), ws.numel(), None, None)
        assert st == 1, (cap, st)
