"""The sampler kernels' CUDA source, run on the CPU.

tests/emu/cuda_emu.h emulates the CUDA primitives the sampler uses (block
barriers, warp shuffles / ballots / reductions, atomics) with one std::thread
per CUDA thread; the library's csrc/sampler.cu is compiled against it with
address and undefined-behaviour sanitizers (bounds, alignment) and run on
seeded inputs.  The sampled tokens must equal the oracle's except at
near-ties, as on the GPU.  Lanes of a warp never run in lockstep here, so a
warp-synchronous assumption in the kernels shows up as a wrong token, and an
out-of-bounds or misaligned access stops the run.  No GPU is needed; this is
a check of the kernels' logic, not a fallback (nothing in the library calls
it)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NEAR = 1e-6


@pytest.fixture(scope="module")
def emu_binary(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    d = tmp_path_factory.mktemp("sampler_emu")
    src = open(os.path.join(ROOT, "paged_kv_decode_pages_gb300", "csrc", "sampler.cu")).read()
    end = src.index("}  // namespace pkv") + len("}  // namespace pkv")
    # every block's shared scratch starts as garbage, as on the device
    dev = src[:end].replace("__shared__ SampSmem sm;",
                            "__shared__ SampSmem sm;\n  emu_poison_shared(&sm, sizeof(sm));")
    (d / "sampler_dev.inc").write_text(dev + "\n")
    exe = d / "sampler_emu"
    cmd = [gxx, "-std=c++20", "-O1", "-g", "-fsanitize=address,undefined",
           "-fno-sanitize-recover=all", "-ffp-contract=off",
           "-I", os.path.join(ROOT, "tests", "emu"), "-I", os.path.join(ROOT, "include"),
           "-I", str(d), os.path.join(ROOT, "tests", "emu", "sampler_emu_main.cpp"),
           "-o", str(exe), "-lpthread"]
    subprocess.run(cmd, check=True, capture_output=True)
    return exe


def _run(exe, tmp_path, x, slots, active, seeds, steps, temp, top_k, top_p, ext=None, zsplit=1,
         single=1):
    """ext: dict of min_p, rep_penalty, rep_window, history [S, cap],
    hist_len, advance (the pkv_seeded_sample_ext settings).  zsplit: launch
    the second CTA per chunk that computes the normaliser (the host does so
    whenever the chunk grid is at most two CTAs per SM).  single: a
    vocabulary of one chunk runs as one kernel (0: as the chunk and finish
    kernels).  Returns
    (out_tok, out_kind, err) and, with ext, also (logprob_raw, logprob_proc,
    hist_len, history, steps) after the call."""
    B, V = x.shape
    S = seeds.shape[0]
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        np.array([B, V, S, 0 if ext is None else 1], np.int32).tofile(f)
        arrs = [(x, np.float32), (slots, np.int32), (active, np.int32), (seeds, np.uint64),
                (steps, np.int64), (temp, np.float32), (top_k, np.int32), (top_p, np.float32)]
        if ext is not None:
            cap = ext["history"].shape[1]
            arrs += [(ext["min_p"], np.float32), (ext["rep_penalty"], np.float32),
                     (ext["rep_window"], np.int32), (np.array([cap]), np.int32),
                     (ext["history"], np.int32), (ext["hist_len"], np.int32),
                     (np.array([int(ext["advance"])]), np.int32)]
        for arr, dt in arrs:
            np.ascontiguousarray(arr, dtype=dt).tofile(f)
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=0", EMU_ZSPLIT=str(int(zsplit)),
               EMU_SINGLE=str(int(single)))
    r = subprocess.run([str(exe), str(inp), str(out)], capture_output=True, text=True, env=env,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    raw = open(out, "rb").read()
    res = np.frombuffer(raw, np.int32, 2 * B + 1)
    base = (res[:B].copy(), res[B:2 * B].copy(), int(res[2 * B]))
    if ext is None:
        return base
    off = 4 * (2 * B + 1)
    lraw = np.frombuffer(raw, np.float32, B, off)
    lproc = np.frombuffer(raw, np.float32, B, off + 4 * B)
    off += 8 * B
    hl = np.frombuffer(raw, np.int32, S, off)
    off += 4 * S
    cap = ext["history"].shape[1]
    hist = np.frombuffer(raw, np.int32, S * cap, off).reshape(S, cap)
    off += 4 * S * cap
    st = np.frombuffer(raw, np.int64, S, off)
    return base + (lraw.copy(), lproc.copy(), hl.copy(), hist.copy(), st.copy())


CASES = [
    # B, V, std, T, k, p, dist
    (3, 1024, 2.0, 0.0, 0, 1.0, "normal"),        # greedy
    (3, 6561, 3.0, 1.0, 25, 0.8, "normal"),       # top-k 25 + top-p, one chunk
    (3, 20000, 1.0, 1.0, 0, 1.0, "normal"),       # keep everything (fp32 Gumbel scores)
    (3, 20000, 1.0, 5.0, 0, 0.95, "normal"),      # top-p crossing past 512 tokens
    (3, 40000, 1.0, 1.0, 200, 0.99, "normal"),    # top-k above the per-chunk candidates
    (3, 40000, 1.0, 1.0, 300, 0.99, "conc"),      # one chunk holds the top-k
    (3, 40000, 1.0, 1.0, 513, 1.0, "normal"),     # general path: top-k > 512
    (2, 151936, 4.0, 0.7, 0, 0.95, "normal"),     # long-context sampler
    (2, 151936, 1.0, 0.5, 0, 0.95, "conc"),       # one chunk holds the top-p set
    # the chunk pass's candidate selection: the lower bound from the thread
    # maxima passes more than 256 composites (radix select instead) ...
    (3, 40000, 1.0, 1.0, 50, 0.9, "stripe"),
    # ... one thread's elements are each chunk's 32 largest ...
    (3, 40000, 1.0, 1.0, 50, 0.95, "thread"),
    # ... a short last chunk (808 tokens) and a chunk with idle warps
    (3, 9000, 1.0, 1.0, 100, 1.0, "normal"),
    (3, 200, 1.0, 1.0, 20, 0.9, "normal"),
    # longer per-warp candidate lists (sorted 64 and 128 to a warp), and a
    # finish that deals 64 union entries to each warp
    (3, 6561, 1.0, 1.0, 128, 0.95, "normal"),
    (3, 6561, 1.0, 1.0, 200, 0.9, "normal"),
    (3, 20000, 1.0, 1.0, 400, 0.97, "normal"),
    (3, 8192, 1.0, 1.0, 230, 0.95, "normal"),   # 90-106 to a warp
    (3, 8192, 1.0, 1.0, 256, 0.95, "normal"),   # over 128 to a warp: radix select
    # lists of one or two slots: the heads' pairwise merge (not the bitonic
    # union), its runs following a token's chunk
    (3, 33000, 1.0, 1.0, 2, 1.0, "normal"),
    (3, 33000, 1.0, 1.0, 1, 1.0, "normal"),
    # rows and last chunks off the 16-byte grid: the chunk copied by
    # cp.async from every thread instead of bulk copies from one
    (3, 20001, 1.0, 1.0, 0, 0.95, "normal"),
    # the finish's bitonic union at its boundaries: 16 lists of 32 slots
    # fill 512 entries exactly (two a thread), 17 lists need 1 024 (four a
    # thread, fifteen lists of padding)
    (2, 131072, 2.0, 0.8, 0, 0.9, "normal"),
    (2, 139264, 2.0, 0.8, 0, 0.9, "normal"),
    # the finish's bitonic merge of the union with lists of 8 and 4 slots
    (3, 40000, 1.0, 1.0, 5, 0.9, "normal"),
    (3, 30000, 2.0, 1.0, 3, 1.0, "normal"),
]


# cases that need the row normaliser, run again with one CTA per chunk (the
# launch for grids larger than two CTAs per SM)
ONE_CTA_CASES = [CASES[3], CASES[7], CASES[8], CASES[12]]


@pytest.mark.parametrize("B,V,std,T,k,p,dist", CASES)
def test_emulated_sampler_matches_oracle(emu_binary, tmp_path, B, V, std, T, k, p, dist):
    _check_case(emu_binary, tmp_path, B, V, std, T, k, p, dist, zsplit=1)


@pytest.mark.parametrize("B,V,std,T,k,p,dist", ONE_CTA_CASES)
def test_emulated_sampler_one_cta_per_chunk(emu_binary, tmp_path, B, V, std, T, k, p, dist):
    _check_case(emu_binary, tmp_path, B, V, std, T, k, p, dist, zsplit=0)


def _check_case(emu_binary, tmp_path, B, V, std, T, k, p, dist, zsplit):
    rng = np.random.default_rng(V + k)
    x = rng.normal(0, std, (B, V)).astype(np.float32)
    if dist == "conc":
        x[:, :8192] += np.float32(6.0)
    elif dist == "stripe":  # a chunk thread's elements (stride 256) share one level
        x = (-(np.arange(V) % 256) * 0.05 + rng.normal(0, 1e-3, (B, V))).astype(np.float32)
    elif dist == "thread":
        x[:, np.arange(V) % 256 == 5] += np.float32(6.0)
    x[0, 3 % V] = -np.inf  # a masked token
    x_ref = x.copy()
    if B > 1:
        # a NaN logit: reported, and ranked like -inf (the oracle sees -inf)
        x[1, (7 * V) // 11] = np.nan
        x_ref[1, (7 * V) // 11] = -np.inf
    B1 = B + 1  # plus one padding row
    x = np.concatenate([x, np.zeros((1, V), np.float32)])
    slots = np.arange(1, B1 + 1, dtype=np.int32)
    slots[-1] = 0
    active = np.ones(B1, np.int32)
    active[-1] = 0
    S = B1 + 1
    seeds = (np.arange(S, dtype=np.uint64) + np.uint64(977))
    steps = np.full(S, 3, np.int64)
    temp = np.full(S, T, np.float32)
    top_k = np.full(S, k, np.int32)
    top_p = np.full(S, p, np.float32)
    got, kind, err = _run(emu_binary, tmp_path, x, slots, active, seeds, steps, temp, top_k, top_p,
                          zsplit=zsplit)
    x_ref = np.concatenate([x_ref, np.zeros((1, V), np.float32)])
    want, wkind, info, _ = oracle.seeded_sample(x_ref, slots, active, seeds, steps.copy(), temp,
                                                   top_k, top_p, advance=False)
    assert err & ~0x10 == 0  # only the logits bit may be set
    if B > 1:
        assert err & 0x10  # the NaN is reported
    near = (info["top2_gap_rel"] < NEAR) | (info["member_margin"] < NEAR)
    mism = got != want
    assert not np.any(mism & ~near), (np.nonzero(mism & ~near), got, want)
    assert got[-1] == 0 and kind[-1] == 0


def _lp_close(got, want):
    """fp32 log-probs: both sides round an fp64 value; the device's raw
    normaliser terms are within 3e-9 of themselves."""
    want = np.asarray(want, np.float32)
    return (np.abs(got.astype(np.float64) - want.astype(np.float64))
            <= 1e-7 + 2 * np.spacing(np.abs(want)).astype(np.float64))


EXT_CASES = [
    # B, V, std, T, k, p, min_p, penalty, window, dist
    (3, 20000, 1.0, 1.0, 0, 1.0, 0.05, 1.0, -1, "normal"),    # min_p keeps > 512: general path
    (3, 20000, 3.0, 1.0, 0, 1.0, 0.1, 1.0, -1, "normal"),     # min_p cut among the candidates
    (3, 6561, 3.0, 1.0, 200, 1.0, 0.3, 1.4, 4, "normal"),     # top-k + min_p, short window
    (3, 20000, 1.0, 1.0, 0, 0.9, 1e-4, 1.0, -1, "normal"),    # min_p boundary past the candidates
    (3, 20000, 2.0, 0.8, 50, 0.9, 0.02, 1.3, 16, "normal"),   # penalty + top-k + min_p + top-p
    (3, 6561, 2.0, 0.0, 0, 1.0, 0.0, 2.0, -1, "normal"),      # greedy with penalty
    (3, 20000, 1.0, 1.0, 0, 1.0, 0.0, 1.2, -1, "normal"),     # keep everything + penalty
    (3, 40000, 1.0, 1.0, 600, 0.95, 0.001, 1.5, 8, "normal"), # general path: top-k > 512
    (2, 151936, 3.0, 0.7, 0, 0.95, 0.01, 1.1, -1, "conc"),    # long-context sampler
]


def _ext_inputs(B, V, std, T, k, p, mp, pen, win, dist):
    rng = np.random.default_rng(V + k + 7)
    x = rng.normal(0, std, (B, V)).astype(np.float32)
    if dist == "conc":
        x[:, :8192] += np.float32(6.0)
    x[0, 3 % V] = -np.inf
    B1 = B + 1
    x = np.concatenate([x, np.zeros((1, V), np.float32)])
    slots = np.arange(1, B1 + 1, dtype=np.int32)
    slots[-1] = 0
    active = np.ones(B1, np.int32)
    active[-1] = 0
    S = B1 + 1
    seeds = (np.arange(S, dtype=np.uint64) + np.uint64(31))
    steps = np.full(S, 5, np.int64)
    temp = np.full(S, T, np.float32)
    top_k = np.full(S, k, np.int32)
    top_p = np.full(S, p, np.float32)
    # histories: each row's recent tokens include its own leaders (so the
    # penalty changes the order) and a repeat; the ring has wrapped
    cap = 24
    history = rng.integers(0, V, (S, cap)).astype(np.int32)
    hist_len = np.full(S, 30, np.int32)
    for b in range(B):
        lead = np.argsort(-x[b], kind="stable")[:6].astype(np.int32)
        s = slots[b]
        for i, t in enumerate(list(lead) + [lead[0]]):
            history[s, (hist_len[s] - 1 - 2 * i) % cap] = t
    ext = dict(min_p=np.full(S, mp, np.float32), rep_penalty=np.full(S, pen, np.float32),
               rep_window=np.full(S, win, np.int32), history=history.copy(),
               hist_len=hist_len.copy(), advance=True)
    return x, slots, active, seeds, steps, temp, top_k, top_p, history, hist_len, ext


@pytest.mark.parametrize("B,V,std,T,k,p,mp,pen,win,dist", EXT_CASES)
def test_emulated_sampler_ext_matches_oracle(emu_binary, tmp_path, B, V, std, T, k, p, mp, pen,
                                             win, dist):
    (x, slots, active, seeds, steps, temp, top_k, top_p, history, hist_len,
     ext) = _ext_inputs(B, V, std, T, k, p, mp, pen, win, dist)
    got, kind, err, lraw, lproc, hl, hist, st = _run(emu_binary, tmp_path, x, slots, active, seeds,
                                                     steps, temp, top_k, top_p, ext)
    w_steps = steps.copy()
    w_hist = history.copy()
    w_len = hist_len.copy()
    want, wraw, wproc, info, _ = oracle.seeded_sample_ext(
        x, slots, active, seeds, w_steps, temp, top_k, top_p, min_p=ext["min_p"],
        rep_penalty=ext["rep_penalty"], rep_window=ext["rep_window"], history=w_hist,
        hist_len=w_len, advance=True)
    assert err & ~0x10 == 0
    near = (info["top2_gap_rel"] < NEAR) | (info["member_margin"] < NEAR)
    mism = got != want
    assert not np.any(mism & ~near), (np.nonzero(mism & ~near), got, want)
    same = ~mism
    assert np.all(_lp_close(lraw[same], wraw[same])), (lraw, wraw)
    assert np.all(_lp_close(lproc[same], wproc[same])), (lproc, wproc)
    assert got[-1] == 0 and lraw[-1] == 0 and lproc[-1] == 0
    np.testing.assert_array_equal(st, w_steps)
    np.testing.assert_array_equal(hl, w_len)
    if not np.any(mism):
        np.testing.assert_array_equal(hist, w_hist)


# The launch shapes the host picks by the grid's size -- a second CTA per
# chunk for the normalisers, one kernel for a vocabulary of one chunk --
# must not change a bit of any output: every output of the default launch
# against the same call launched the other way (tokens, kinds, both
# log-probs' bits, rings, lengths, step counters, the error word).
SHAPE_CASES = [
    (EXT_CASES[2], "single"),   # 6 561 tokens, penalty, log-probs
    (EXT_CASES[5], "single"),   # greedy with penalty
    (EXT_CASES[4], "zsplit"),   # 20 000 tokens: raw log-prob in the second CTA
    (EXT_CASES[3], "zsplit"),
    ((2, 151936, 3.0, 0.7, 0, 0.95, 0.0, 1.0, -1, "normal"), "zsplit"),  # top-p normaliser
]


@pytest.mark.parametrize("case,shape", SHAPE_CASES)
def test_emulated_launch_shapes_give_the_same_bits(emu_binary, tmp_path, case, shape):
    outs = []
    for alt in (False, True):
        (x, slots, active, seeds, steps, temp, top_k, top_p, history, hist_len,
         ext) = _ext_inputs(*case)
        kw = {"zsplit": 0} if (alt and shape == "zsplit") else {}
        if alt and shape == "single":
            kw = {"single": 0}
        outs.append(_run(emu_binary, tmp_path, x, slots, active, seeds, steps, temp, top_k,
                         top_p, ext, **kw))
    a, b = outs
    for u, v in zip(a, b):
        u, v = np.asarray(u), np.asarray(v)
        assert u.dtype == v.dtype and u.shape == v.shape
        assert u.tobytes() == v.tobytes(), (shape, u, v)
