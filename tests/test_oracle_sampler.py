"""Pins of the oracle's seeded sampler, Philox stream and frame loop against
things other than itself: numpy's Philox4x64-10 raw words, the Gumbel
distribution's mean and variance, numpy.argmax, kept sets enumerated by
brute force on tiny vocabularies, hand-built boundary cases, and a
chi-square test of Gumbel-max frequencies against the renormalised kept-set
probabilities.

Semantics: "Supported Models" (mstar docs), "Fish Audio S2-Pro notes"
(temperature first, then top-k / top-p over the tempered probabilities; the
top-p boundary keeps the token that carries the running total past top-p),
"Chatterbox notes" (temperature under 1e-5 is greedy, top-k of the whole
vocabulary or more is no filter), "Adding a Model" (vox-serve docs), "How a
program runs" (per-request seeds) and "2. The program" (a different salt per
sampling call; stop_tokens / audio_tokens); MOSS-TTS-Local on SGLang-Omni
(mosi.cn blog), model section (12 codebooks, each fed back before the next).
"""
import math

import numpy as np
import pytest
from scipy import stats

import oracle


# ---------------------------------------------------------------------------
# Philox4x64-10 and the Gumbel noise
# ---------------------------------------------------------------------------
def _inc(ctr):
    c = [int(x) for x in ctr]
    for i in range(4):
        c[i] = (c[i] + 1) % (1 << 64)
        if c[i]:
            break
    return np.array(c, np.uint64)


@pytest.mark.parametrize("key,ctr", [
    ((0, 0), (0, 0, 0, 0)),
    ((1, 2), (0, 0, 0, 0)),
    ((12345, 7), (41, 3, 0, 0)),
    ((2**64 - 1, 2**63 + 5), (2**64 - 1, 2**64 - 1, 9, 0)),
    ((0xDEADBEEF, 0), (2**64 - 1, 0, 0, 0)),
])
def test_philox_matches_numpy_raw_words(key, ctr):
    key = np.array(key, np.uint64)
    ctr = np.array(ctr, np.uint64)
    # numpy's Philox bumps its 256-bit counter before producing each block
    want = np.random.Philox(counter=ctr, key=key).random_raw(4)
    got = oracle.philox4x64_10(key, _inc(ctr))
    np.testing.assert_array_equal(got, want)


def _dec(ctr):
    c = [int(x) for x in ctr]
    for i in range(4):
        borrow = c[i] == 0
        c[i] = (c[i] - 1) % (1 << 64)
        if not borrow:
            break
    return np.array(c, np.uint64)


def test_uniform_uses_word0_and_is_strictly_inside_unit_interval():
    for seed, salt, tok, step in [(0, 0, 0, 0), (9, 1, 151935, 77), (2**63, 12, 5, 2**40)]:
        key = np.array([seed, salt], np.uint64)
        ctr = np.array([tok, step, 0, 0], np.uint64)
        words = np.random.Philox(counter=_dec(ctr), key=key).random_raw(4)
        u = oracle.uniform(seed, salt, tok, step)
        assert 0.0 < u < 1.0
        assert u == (2 * (int(words[0]) >> 12) + 1) * 2.0 ** -53
    # the extremes of the mapping are exact and strictly inside (0, 1)
    assert (2 * 0 + 1) * 2.0 ** -53 > 0
    assert (2 * (2**52 - 1) + 1) * 2.0 ** -53 < 1.0


def test_gumbel_moments():
    """Standard Gumbel: mean = Euler-Mascheroni gamma, variance = pi^2 / 6."""
    g = np.array([oracle.gumbel(3, 1, t, 0) for t in range(200000)])
    assert abs(g.mean() - np.euler_gamma) < 0.01
    assert abs(g.var() - math.pi ** 2 / 6) < 0.02
    # Kolmogorov-Smirnov against scipy's Gumbel
    assert stats.kstest(g[:20000], "gumbel_r").pvalue > 1e-4


# ---------------------------------------------------------------------------
# Greedy conventions
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("temp", [0.0, 1e-6, 1e-5, -1.0])
def test_greedy_is_numpy_argmax(temp):
    rng = np.random.default_rng(0)
    for _ in range(20):
        x = rng.integers(-3, 3, size=37).astype(np.float32)  # many exact ties
        tok, info = oracle.sample_row(x, seed=1, step=2, salt=0, temperature=temp, top_k=0, top_p=1.0)
        assert tok == int(np.argmax(x)) and info["greedy"] == 1


def test_top_k_one_and_tiny_top_p_are_argmax_for_any_seed():
    rng = np.random.default_rng(1)
    for i in range(50):
        x = rng.normal(0, 2, size=300).astype(np.float32)
        x[rng.integers(0, 300)] = x.max()  # a tie at the top: lowest id wins
        a = int(np.argmax(x))
        assert oracle.sample_row(x, i, i, 0, 0.7, 1, 1.0)[0] == a
        assert oracle.sample_row(x, i, i, 3, 1.3, 0, 1e-9)[0] == a


# ---------------------------------------------------------------------------
# Kept sets by brute force
# ---------------------------------------------------------------------------
def _brute_kept(x32, temp, top_k, top_p):
    """Kept set from pairwise comparisons (no sort): token i precedes j when
    x_i > x_j, or x_i == x_j and i < j."""
    V = len(x32)
    x = [float(v) / float(np.float32(temp)) for v in x32]
    before = lambda j, i: x[j] > x[i] or (x[j] == x[i] and j < i)
    rank = [sum(before(j, i) for j in range(V)) for i in range(V)]
    K = top_k if 0 < top_k < V else V
    surv = [i for i in range(V) if rank[i] < K]
    if top_p >= 1.0:
        return set(surv), None
    m = max(x)
    e = {i: math.exp(x[i] - m) for i in surv}
    Z = sum(e[i] for i in sorted(surv, key=lambda i: rank[i]))
    kept = set()
    for i in surv:
        S = sum(e[j] for j in sorted(surv, key=lambda j: rank[j]) if rank[j] < rank[i])
        if rank[i] == 0 or S < float(np.float32(top_p)) * Z:
            kept.add(i)
    probs = {i: e[i] for i in kept}
    return kept, probs


@pytest.mark.parametrize("V", [2, 3, 5, 8])
def test_kept_set_count_matches_brute_force(V):
    rng = np.random.default_rng(V)
    for trial in range(300):
        x = rng.normal(0, 1.5, size=V).astype(np.float32)
        if trial % 5 == 0:
            x[rng.integers(0, V)] = x[rng.integers(0, V)]  # exact tie
        temp = float(rng.choice([0.5, 1.0, 2.0]))
        k = int(rng.integers(0, V + 2))
        p = float(rng.choice([0.3, 0.6, 0.9, 1.0]))
        kept, _ = _brute_kept(x, temp, k, p)
        tok, info = oracle.sample_row(x, trial, 0, 0, temp, k, p)
        assert info["n_kept"] == len(kept)
        assert tok in kept


def test_top_p_boundary_prefix_exactly_p_drops_the_next_token():
    # four equal logits: q = 1/4 each; p = 1/2.  The second token carries the
    # running total from 1/4 to 1/2 and is kept; the third would start at
    # exactly 1/2 = p and is dropped.  Ties go to the lower id.
    x = np.zeros(4, np.float32)
    seen = set()
    for step in range(400):
        tok, info = oracle.sample_row(x, 5, step, 0, 1.0, 0, 0.5)
        assert info["n_kept"] == 2
        seen.add(tok)
    assert seen == {0, 1}


def test_top_p_keeps_the_crossing_token():
    # softmax probabilities about 0.5, 0.25, 0.125, 0.125; with p = 0.6 the
    # second token takes the running total from 0.5 past 0.6 and is kept, the
    # third starts above p and is dropped
    x = np.array([3 * math.log(2), 2 * math.log(2), math.log(2), math.log(2)], np.float32)
    kept, _ = _brute_kept(x, 1.0, 0, 0.6)
    assert kept == {0, 1}  # 0.5 < 0.6 so the second token (crossing) is kept
    for step in range(200):
        tok, info = oracle.sample_row(x, 1, step, 0, 1.0, 0, 0.6)
        assert info["n_kept"] == 2 and tok in kept


def test_top_k_tie_at_the_cut_goes_to_lower_ids():
    x = np.array([5, 3, 3, 3, 1], np.float32)
    seen = set()
    for step in range(300):
        tok, info = oracle.sample_row(x, 2, step, 0, 4.0, 2, 1.0)
        assert info["n_kept"] == 2
        seen.add(tok)
    assert seen == {0, 1}


def test_top_k_of_whole_vocab_or_more_is_no_filter():
    x = np.random.default_rng(3).normal(0, 1, 10).astype(np.float32)
    for k in (0, 10, 11, 1000):
        assert oracle.sample_row(x, 1, 0, 0, 1.0, k, 1.0)[1]["n_kept"] == 10


@pytest.mark.parametrize("top_k,top_p,temp", [(0, 1.0, 1.0), (5, 1.0, 0.7), (0, 0.8, 1.3), (6, 0.7, 0.9)])
def test_gumbel_max_frequencies_chi_square(top_k, top_p, temp):
    """P(sample = i) equals the renormalised kept-set probability of i."""
    x = np.random.default_rng(42).normal(0, 1.0, 16).astype(np.float32)
    kept, probs = _brute_kept(x, temp, top_k, top_p)
    if probs is None:
        xs = np.array([float(v) / float(np.float32(temp)) for v in x])
        e = np.exp(xs - xs.max())
        probs = {i: e[i] for i in kept}
    ids = sorted(kept)
    p = np.array([probs[i] for i in ids])
    p /= p.sum()
    n = 40000
    counts = np.zeros(16, np.int64)
    for step in range(n):
        counts[oracle.sample_row(x, 77, step, 9, temp, top_k, top_p)[0]] += 1
    assert counts[[i for i in range(16) if i not in kept]].sum() == 0
    chi = stats.chisquare(counts[ids], p * n)
    assert chi.pvalue > 1e-4, chi


def test_seed_salt_step_each_change_the_stream():
    x = np.zeros(1000, np.float32)  # uniform over 1000 tokens
    base = [oracle.sample_row(x, 1, s, 0, 1.0, 0, 1.0)[0] for s in range(30)]
    assert base == [oracle.sample_row(x, 1, s, 0, 1.0, 0, 1.0)[0] for s in range(30)]
    assert base != [oracle.sample_row(x, 2, s, 0, 1.0, 0, 1.0)[0] for s in range(30)]
    assert base != [oracle.sample_row(x, 1, s, 1, 1.0, 0, 1.0)[0] for s in range(30)]
    assert base != [oracle.sample_row(x, 1, s + 1, 0, 1.0, 0, 1.0)[0] for s in range(30)]


def test_kinds_stop_takes_precedence():
    stops = [7, 100]
    assert oracle.token_kind(7, stops, 0, 50) == oracle.KIND_STOP
    assert oracle.token_kind(100, stops, 0, 200) == oracle.KIND_STOP
    assert oracle.token_kind(49, stops, 0, 50) == oracle.KIND_AUDIO
    assert oracle.token_kind(50, stops, 0, 50) == oracle.KIND_OTHER
    assert oracle.token_kind(3, [], 5, 9) == oracle.KIND_OTHER


def test_batched_sampler_padding_and_advance():
    rng = np.random.default_rng(4)
    B, V = 6, 64
    x = rng.normal(0, 2, (B, V)).astype(np.float32)
    slots = np.array([1, 2, 0, 3, 4, 0], np.int32)
    active = np.array([1, 1, 0, 1, 1, 0], np.int32)
    seeds = np.arange(5, dtype=np.uint64) * 11
    steps = np.array([100, 3, 4, 5, 6], np.int64)
    T = np.full(5, 0.9, np.float32)
    K = np.full(5, 10, np.int32)
    P = np.full(5, 0.9, np.float32)
    tok, kind, info, bad = oracle.seeded_sample(x, slots, active, seeds, steps, T, K, P, salt=0,
                                                advance=True, stop_tokens=[5], audio_lo=10,
                                                audio_hi=40)
    assert bad == 0
    assert list(steps) == [100, 4, 5, 6, 7]  # dummy slot 0 untouched
    for b in range(B):
        if not active[b]:
            assert tok[b] == 0 and kind[b] == oracle.KIND_OTHER
            continue
        s = slots[b]
        t1, _ = oracle.sample_row(x[b], seeds[s], steps[s] - 1, 0, T[s], K[s], P[s])
        assert tok[b] == t1
        assert kind[b] == oracle.token_kind(t1, [5], 10, 40)


# ---------------------------------------------------------------------------
# Frame loop
# ---------------------------------------------------------------------------
def _frame_inputs(seed=0, n_cb=12, B=3, V=64):
    rng = np.random.default_rng(seed)
    base = rng.normal(0, 3, (n_cb, B, V)).astype(np.float32)
    fb = rng.normal(0, 1, (n_cb, V, V)).astype(np.float32)
    slots = np.array([1, 0, 2][:B], np.int32)
    active = np.array([1, 0, 1][:B], np.int32)
    seeds = np.array([0, 21, 22], np.uint64)
    T = np.full(3, 0.9, np.float32)
    K = np.full(3, 8, np.int32)
    P = np.full(3, 0.9, np.float32)
    return base, fb, slots, active, seeds, T, K, P


def test_frame_without_feedback_equals_independent_salted_samples():
    base, fb, slots, active, seeds, T, K, P = _frame_inputs()
    steps = np.array([0, 7, 9], np.int64)
    codes, kind, _, bad = oracle.codebook_frame_sample(base, None, slots, active, seeds, steps, T, K, P)
    assert bad == 0 and list(steps) == [0, 8, 10]
    for b in range(3):
        if not active[b]:
            assert np.all(codes[b] == 0) and kind[b] == oracle.KIND_OTHER
            continue
        s = slots[b]
        want = [oracle.sample_row(base[j, b], seeds[s], steps[s] - 1, 1 + j, T[s], K[s], P[s])[0]
                for j in range(12)]
        assert list(codes[b]) == want and kind[b] == oracle.KIND_AUDIO


def test_frame_feedback_wiring():
    """Codebook j > 0 samples base[j] + fb[j][code_{j-1}], added in fp32."""
    base, fb, slots, active, seeds, T, K, P = _frame_inputs(seed=1)
    steps = np.array([0, 3, 4], np.int64)
    codes, _, _, _ = oracle.codebook_frame_sample(base, fb, slots, active, seeds, steps.copy(), T, K, P)
    for b in (0, 2):
        s = slots[b]
        prev = None
        for j in range(12):
            row = base[j, b] if j == 0 else (base[j, b] + fb[j, prev]).astype(np.float32)
            prev = oracle.sample_row(row, seeds[s], steps[s], 1 + j, T[s], K[s], P[s])[0]
            assert codes[b, j] == prev
    # the feedback matters: zero it and the codes change somewhere
    codes0, _, _, _ = oracle.codebook_frame_sample(base, np.zeros_like(fb), slots, active, seeds,
                                                   steps.copy(), T, K, P)
    codes_none, _, _, _ = oracle.codebook_frame_sample(base, None, slots, active, seeds,
                                                       steps.copy(), T, K, P)
    np.testing.assert_array_equal(codes0, codes_none)
    assert np.any(codes0 != codes)


# ---------------------------------------------------------------------------
# Full frame: the stop/continue sample on channel 0, then the codebooks
# ---------------------------------------------------------------------------
STOP = 2  # the stop token of a 4-token control vocabulary in these tests


def _ctrl(bias_stop):
    """Control logits [3, 4]; bias_stop[b] is added to the stop token's."""
    rng = np.random.default_rng(17)
    c = rng.normal(0, 1.0, (3, 4)).astype(np.float32)
    c[:, STOP] += np.asarray(bias_stop, np.float32)
    return c


def test_full_frame_channel0_is_the_salt0_sample_and_gates_the_codes():
    base, fb, slots, active, seeds, T, K, P = _frame_inputs(seed=2)
    ctrl = _ctrl([30.0, 0.0, -np.inf])  # row 0 must stop, row 2 cannot
    steps = np.array([0, 3, 4], np.int64)
    rows, kind, _, bad = oracle.frame_sample(ctrl, STOP, base, fb, slots, active, seeds,
                                             steps, T, K, P)
    assert bad == 0 and list(steps) == [0, 4, 5]  # once per frame, stopped or not
    codes, _, _, _ = oracle.codebook_frame_sample(base, fb, slots, active, seeds,
                                                  np.array([0, 3, 4], np.int64), T, K, P)
    assert np.all(rows[1] == 0) and kind[1] == oracle.KIND_OTHER  # padding row
    for b in (0, 2):
        s = slots[b]
        c0 = oracle.sample_row(ctrl[b], seeds[s], steps[s] - 1, 0, T[s], K[s], P[s])[0]
        assert rows[b, 0] == c0
    assert rows[0, 0] == STOP and kind[0] == oracle.KIND_STOP
    assert np.all(rows[0, 1:] == oracle.CODE_PAD)
    assert rows[2, 0] != STOP and kind[2] == oracle.KIND_AUDIO
    np.testing.assert_array_equal(rows[2, 1:], codes[2])


def test_full_frame_that_never_stops_is_the_codebook_frame():
    base, fb, slots, active, seeds, T, K, P = _frame_inputs(seed=3)
    ctrl = _ctrl([-np.inf] * 3)
    s1, s2 = np.array([0, 5, 6], np.int64), np.array([0, 5, 6], np.int64)
    rows, kind, _, _ = oracle.frame_sample(ctrl, STOP, base, fb, slots, active, seeds, s1, T, K, P)
    codes, ckind, _, _ = oracle.codebook_frame_sample(base, fb, slots, active, seeds, s2, T, K, P)
    np.testing.assert_array_equal(rows[:, 1:], codes)
    np.testing.assert_array_equal(kind, ckind)
    np.testing.assert_array_equal(s1, s2)
    assert np.all(rows[[0, 2], 0] != STOP)


def test_full_frame_that_always_stops_is_a_pad_row():
    base, fb, slots, active, seeds, T, K, P = _frame_inputs(seed=4)
    ctrl = np.full((3, 4), -np.inf, np.float32)
    ctrl[:, STOP] = 0.0  # the only finite control logit
    steps = np.array([0, 1, 2], np.int64)
    rows, kind, _, _ = oracle.frame_sample(ctrl, STOP, base, fb, slots, active, seeds, steps,
                                           T, K, P)
    for b in (0, 2):
        assert list(rows[b]) == [STOP] + [oracle.CODE_PAD] * 12 and kind[b] == oracle.KIND_STOP
    assert list(steps) == [0, 2, 3]


# ---------------------------------------------------------------------------
# Further controls: repetition penalty, min_p; raw / processed log-probs
# ---------------------------------------------------------------------------
def test_ext_with_the_controls_off_is_the_base_sampler():
    rng = np.random.default_rng(31)
    for trial in range(40):
        x = rng.normal(0, 2, 300).astype(np.float32)
        k, p, T = [(0, 1.0, 1.0), (20, 0.9, 0.7), (0, 0.5, 1.3), (5, 1.0, 0.8)][trial % 4]
        a = oracle.sample_row(x, 7, trial, 3, T, k, p)[0]
        b = oracle.sample_row_ext(x, 7, trial, 3, T, k, p, min_p=0.0, rep_penalty=1.0,
                                  pen_tokens=[1, 2, 3])[0]
        assert a == b


def test_raw_logprob_is_scipy_log_softmax_of_the_unprocessed_logits():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(32)
    for trial in range(20):
        x = rng.normal(0, 3, 500).astype(np.float32)
        tok, info = oracle.sample_row_ext(x, 9, trial, 0, 0.8, 40, 0.9, min_p=0.05,
                                          rep_penalty=1.7, pen_tokens=list(range(0, 500, 7)))
        want = scipy_special.log_softmax(x.astype(np.float64))[tok]
        assert abs(info["logprob_raw"] - want) < 1e-12


def test_processed_logprob_closed_forms():
    rng = np.random.default_rng(33)
    x = rng.normal(0, 2, 64).astype(np.float32)
    # no processing at T = 1: the raw log-prob
    _, info = oracle.sample_row_ext(x, 1, 2, 0, 1.0, 0, 1.0)
    assert abs(info["logprob_proc"] - info["logprob_raw"]) < 1e-12
    # a point mass: greedy, top-k 1, min_p 1 without ties
    for kw in (dict(temperature=0.0, top_k=0), dict(temperature=1.0, top_k=1),
               dict(temperature=1.0, top_k=0, min_p=1.0)):
        T, k = kw.pop("temperature"), kw.pop("top_k")
        _, info = oracle.sample_row_ext(x, 1, 2, 0, T, k, 1.0, **kw)
        assert info["logprob_proc"] == 0.0 and info["n_kept"] == 1


@pytest.mark.parametrize("T,k,p,min_p,pen", [(1.0, 0, 1.0, 0.1, 1.0), (0.8, 6, 0.9, 0.05, 1.8),
                                             (1.5, 0, 0.7, 0.2, 0.6)])
def test_processed_logprob_is_the_sampling_distribution(T, k, p, min_p, pen):
    """Gumbel-max frequencies over many steps against exp(logprob_proc)
    reported for each drawn token (a chi-square over the kept tokens)."""
    scipy_stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(34)
    x = rng.normal(0, 0.5, 12).astype(np.float32)
    pen_tokens = [0, 3, 3, 7]
    n = 20000
    counts = {}
    prob = {}
    for step in range(n):
        tok, info = oracle.sample_row_ext(x, 5, step, 0, T, k, p, min_p=min_p, rep_penalty=pen,
                                          pen_tokens=pen_tokens)
        counts[tok] = counts.get(tok, 0) + 1
        lp = info["logprob_proc"]
        if tok in prob:
            assert abs(prob[tok] - lp) < 1e-12  # the same distribution every step
        prob[tok] = lp
    toks = sorted(counts)
    assert len(toks) >= 3, toks  # the filters leave a distribution to test
    p_obs = np.array([counts[t] for t in toks], float)
    p_exp = np.exp(np.array([prob[t] for t in toks]))
    assert abs(p_exp.sum() - 1.0) < 1e-3  # every kept token was drawn
    chi2, pv = scipy_stats.chisquare(p_obs, p_exp / p_exp.sum() * n)
    assert pv > 1e-4, (pv, toks)


def test_repetition_penalty_rule_closed_form():
    """Greedy picks expose the penalised logits: positive / pen, negative
    * pen, zero unchanged, once per distinct id, ids outside [0, V) ignored."""
    x = np.array([3.0, 2.5, -1.0, -1.2, 0.0, -4.0], np.float32)
    g = lambda pen, toks: oracle.sample_row_ext(x, 0, 0, 0, 0.0, 0, 1.0, rep_penalty=pen,
                                                pen_tokens=toks)[0]
    assert g(1.5, [0]) == 1                  # 3 / 1.5 = 2 < 2.5
    assert g(1.1, [0]) == 0                  # 3 / 1.1 > 2.5
    assert g(1.1, [0, 0, 0, 0]) == 0         # not compounded by repeats
    y = np.array([-1.0, -1.2, -5.0], np.float32)
    gy = lambda pen, toks: oracle.sample_row_ext(y, 0, 0, 0, 0.0, 0, 1.0, rep_penalty=pen,
                                                 pen_tokens=toks)[0]
    assert gy(1.3, [0]) == 1                 # -1.3 < -1.2
    assert gy(1.3, [0, -1, 7]) == 1          # out-of-range ids are ignored
    z = np.array([0.0, -0.5], np.float32)
    assert oracle.sample_row_ext(z, 0, 0, 0, 0.0, 0, 1.0, rep_penalty=50.0,
                                 pen_tokens=[0])[0] == 0  # 0 stays 0


def test_min_p_keeps_exactly_the_ties_with_the_maximum_at_one():
    x = np.array([1.0, 2.0, 2.0, 1.999, 2.0], np.float32)
    seen = set()
    for step in range(300):
        tok, info = oracle.sample_row_ext(x, 3, step, 0, 1.0, 0, 1.0, min_p=1.0)
        assert info["n_kept"] == 3
        seen.add(tok)
    assert seen == {1, 2, 4}


def test_seeded_sample_ext_history_ring_and_window():
    V = 16
    x = np.zeros((2, V), np.float32)
    x[:, 5] = 2.0
    x[:, 9] = 1.9
    slots = np.array([1, 2], np.int32)
    active = np.array([1, 1], np.int32)
    seeds = np.array([0, 11, 12], np.uint64)
    T = np.zeros(3, np.float32)  # greedy: the penalty decides
    K = np.zeros(3, np.int32)
    P = np.ones(3, np.float32)
    pen = np.full(3, 2.0, np.float32)
    win = np.array([-1, 1, 1], np.int32)
    cap = 4
    hist = np.zeros((3, cap), np.int32)
    hlen = np.zeros(3, np.int32)
    # slot 1: history ring [5, 3, 3, 3, 3] (len 5 wraps): window 1 sees only the last 3
    for t in (5, 3, 3, 3, 3):
        hist[1, hlen[1] % cap] = t
        hlen[1] += 1
    # slot 2: history [5, 1, 2]: window 1 sees only the newest, 2 (not 5)
    for t in (5, 1, 2):
        hist[2, hlen[2] % cap] = t
        hlen[2] += 1
    steps = np.zeros(3, np.int64)
    tok, lraw, lproc, info, bad = oracle.seeded_sample_ext(x, slots, active, seeds, steps, T, K, P,
                                                           rep_penalty=pen, rep_window=win,
                                                           history=hist, hist_len=hlen)
    assert bad == 0 and list(tok) == [5, 5]
    assert list(hlen) == [0, 6, 4] and hist[1, 5 % cap] == 5 and hist[2, 3] == 5
    # with the whole history in the window slot 2 avoids 5
    hist2, hlen2 = np.zeros((3, cap), np.int32), np.zeros(3, np.int32)
    for t in (5, 1, 2):
        hist2[2, hlen2[2] % cap] = t
        hlen2[2] += 1
    tok2, _, _, _, _ = oracle.seeded_sample_ext(x, slots, active, seeds, np.zeros(3, np.int64),
                                                T, K, P, rep_penalty=pen,
                                                rep_window=np.array([-1, 1, -1], np.int32),
                                                history=hist2, hist_len=hlen2)
    assert tok2[1] == 9
    assert list(steps) == [0, 1, 1]
    assert np.all(lproc == 0.0)  # greedy


# ---------------------------------------------------------------------------
# The exact draw: which token id and step each kept token's noise comes from
# ---------------------------------------------------------------------------
def _numpy_gumbel(seed, salt, token, step):
    """Gumbel noise of (seed, salt, token, step) from numpy's own Philox4x64-10
    (key = (seed, salt), counter = (token, step, 0, 0)), word 0 mapped to
    u = (2 * (w >> 12) + 1) * 2^-53, then -log(-log u)."""
    key = np.array([seed, salt], np.uint64)
    ctr = np.array([token, step, 0, 0], np.uint64)
    w = int(np.random.Philox(counter=_dec(ctr), key=key).random_raw(4)[0])
    u = (2 * (w >> 12) + 1) * 2.0 ** -53
    return -math.log(-math.log(u))


def _expected_draw(x32, seed, salt, step, temp, top_k, top_p):
    """Gumbel-max over the brute-force kept set, the noise of each kept token
    drawn for its own id at the request's step; ties to the lowest id.
    Returns (token, gap between the two best scores)."""
    kept, _ = _brute_kept(x32, temp, top_k, top_p)
    T = float(np.float32(temp))
    scores = sorted(((float(x32[i]) / T + _numpy_gumbel(seed, salt, i, step), i) for i in kept),
                    key=lambda si: (-si[0], si[1]))
    gap = scores[0][0] - scores[1][0] if len(scores) > 1 else math.inf
    return scores[0][1], gap


@pytest.mark.parametrize("V", [6, 16])
def test_sampled_token_is_the_gumbel_argmax_of_numpy_philox_noise(V):
    """"Adding a Model", "How a program runs" (draws from per-request seeds)
    and "2. The program" (a salt per sampling call): the token equals the
    argmax of x_i + g(seed, salt, i, step) over the kept set, with g built
    here from numpy's Philox words, for top-k / top-p on and off.  Noise
    indexed by the sorted rank, or with step and token swapped in the
    counter, picks another token on many of these draws."""
    rng = np.random.default_rng(100 + V)
    settings = [(1.0, 0, 1.0), (0.7, 4, 1.0), (1.3, 0, 0.8), (0.9, 5, 0.85)]
    checked = 0
    for trial in range(160):
        x = rng.normal(0, 1.0, V).astype(np.float32)
        temp, k, p = settings[trial % len(settings)]
        seed = int(rng.integers(0, 2**63)) * (1 + trial % 2)
        salt = int(rng.integers(0, 13))
        step = int(rng.integers(0, 5000))
        want, gap = _expected_draw(x, seed, salt, step, temp, k, p)
        if gap < 1e-9:
            continue  # an exact or last-ulp tie between two scores decides nothing
        tok, _ = oracle.sample_row(x, seed, step, salt, temp, k, p)
        assert tok == want, (trial, seed, salt, step, temp, k, p)
        tok_ext, _ = oracle.sample_row_ext(x, seed, step, salt, temp, k, p, min_p=0.0,
                                           rep_penalty=1.0, pen_tokens=[])
        assert tok_ext == want
        checked += 1
    assert checked >= 150


def test_batched_and_frame_draws_use_the_slot_step_and_call_salt():
    """The batched sampler draws row b at its slot's step (before the
    advance) with the call's salt; a frame's codebook j draws with salt 1 + j
    at the frame's step: both against numpy-Philox noise."""
    rng = np.random.default_rng(7)
    V = 12
    x = rng.normal(0, 1.0, (3, V)).astype(np.float32)
    slots = np.array([2, 1, 3], np.int32)
    active = np.ones(3, np.int32)
    seeds = np.array([0, 91, 92, 93], np.uint64)
    steps = np.array([0, 40, 7, 1234], np.int64)
    T = np.full(4, 0.8, np.float32)
    K = np.zeros(4, np.int32)
    P = np.ones(4, np.float32)
    before = steps.copy()
    tok, _, _, bad = oracle.seeded_sample(x, slots, active, seeds, steps, T, K, P, salt=5,
                                          advance=True)
    assert bad == 0
    for b in range(3):
        s = slots[b]
        want, gap = _expected_draw(x[b], int(seeds[s]), 5, int(before[s]), 0.8, 0, 1.0)
        assert gap > 1e-9 and tok[b] == want
    base = rng.normal(0, 1.0, (12, 3, V)).astype(np.float32)
    steps2 = before.copy()
    codes, _, _, bad = oracle.codebook_frame_sample(base, None, slots, active, seeds, steps2,
                                                    T, K, P)
    assert bad == 0
    for b in range(3):
        s = slots[b]
        for j in range(12):
            want, gap = _expected_draw(base[j, b], int(seeds[s]), 1 + j, int(before[s]), 0.8, 0,
                                       1.0)
            if gap > 1e-9:
                assert codes[b, j] == want, (b, j)
