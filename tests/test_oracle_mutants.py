"""The pins are strong enough: each plausible mistake below, planted in a copy
of the oracle's C source and compiled on the CPU, makes at least one pin of
tests/test_oracle_attention.py, tests/test_oracle_prefill.py or
tests/test_oracle_sampler.py fail.  (The
real oracle is untouched; the mutant is loaded only inside this test.)"""
import os
import tempfile

import pytest

import oracle
import test_oracle_attention as TA
import test_oracle_prefill as TP
import test_oracle_sampler as TS

# (name, original text, planted mistake)
MUTANTS = [
    ("gqa head mapping by modulo", "const int n = seq_lens[b];\n    const int g = h / group;",
     "const int n = seq_lens[b];\n    const int g = h % num_kv_heads;"),
    ("prefill gqa head mapping by modulo",
     "const int n = pos[t] + 1; /* keys [0, pos] */\n    const int g = h / group;",
     "const int n = pos[t] + 1; /* keys [0, pos] */\n    const int g = h % num_kv_heads;"),
    ("softmax scale dropped", "s[t] = sm_scale * dot;", "s[t] = dot;"),
    ("keys read from the V half", "pg, 0, t % page_size, g);", "pg, 1, t % page_size, g);"),
    ("values read from the K half", "pg, 1, t % page_size, g);", "pg, 0, t % page_size, g);"),
    ("softmax not normalised", "double p = s[t] / z;", "double p = s[t];"),
    ("lse without the max", "lse[bh] = m + log(z);", "lse[bh] = log(z);"),
    ("append slot off by one", "slot = pos % page_size;\n      if (page < 0",
     "slot = (pos + 1) % page_size;\n      if (page < 0"),
    ("philox xors the wrong high half", "uint64_t y0 = hi1 ^ x1 ^ k0;",
     "uint64_t y0 = hi0 ^ x1 ^ k0;"),
    ("philox bumps k1 by the wrong constant", "k1 += PHILOX_W1;", "k1 += PHILOX_W0;"),
    ("uniform from word 1", "uint64_t j = w[0] >> 12;", "uint64_t j = w[1] >> 12;"),
    ("gumbel sign flipped", "return -log(-log(u));", "return log(-log(u));"),
    ("top-p boundary inclusive", "if (r == 0 || S < pz) {", "if (r == 0 || S <= pz) {"),
    ("top-p drops the crossing token", "if (r == 0 || S < pz) {",
     "if (r == 0 || S + e[r] < pz) {"),
    ("ties to the higher id", "return (p->id > q->id) - (p->id < q->id);",
     "return (p->id < q->id) - (p->id > q->id);"),
    ("top-k keeps one too many", "int K = (top_k > 0 && top_k < V) ? top_k : V;",
     "int K = (top_k > 0 && top_k < V) ? top_k + 1 : V;"),
    ("greedy only at zero temperature", "if (!(temperature > 1e-5f)) {",
     "if (!(temperature > 0.0f)) {"),
    ("frame salt starts at 0", "step, (uint32_t)(1 + j),", "step, (uint32_t)(j),"),
    ("frame feedback from the previous codebook's table",
     "const float *fj = fb + ((int64_t)j * V + prev) * V;",
     "const float *fj = fb + ((int64_t)(j - 1) * V + prev) * V;"),
    ("control sample with a codebook's salt",
     "r[0] = pkvo_sample_row(ctrl + (int64_t)b * Vc, Vc, seeds[s], steps[s], 0u,",
     "r[0] = pkvo_sample_row(ctrl + (int64_t)b * Vc, Vc, seeds[s], steps[s], 1u,"),
    ("a stop leaves the codes unpadded", "for (int j = 1; j < W; ++j) r[j] = PKVO_CODE_PAD;",
     "for (int j = 1; j < W; ++j) r[j] = 0;"),
    ("a stop still samples the codes", "      out_kind[b] = PKVO_KIND_STOP;\n      continue;",
     "      out_kind[b] = PKVO_KIND_STOP;"),
    ("penalty multiplies positive logits", "pl[t] = pl[t] > 0.0f ? pl[t] / rep_penalty : pl[t] * rep_penalty;",
     "pl[t] = pl[t] * rep_penalty;"),
    ("penalty compounds repeats", "if (t < 0 || t >= V || done[t]) continue;",
     "if (t < 0 || t >= V) continue;"),
    ("min_p keeps strictly above", "while (Kp < K && e[Kp] >= (double)min_p) ++Kp;",
     "while (Kp < K && e[Kp] > (double)min_p) ++Kp;"),
    ("top-p ignores min_p", "  for (int r = 0; r < Kp; ++r) S += e[r];\n  if (top_p < 1.0f) {",
     "  for (int r = 0; r < K; ++r) S += e[r];\n  if (top_p < 1.0f) {"),
    ("raw log-prob from the penalised logits", "  for (int i = 0; i < V; ++i) zraw += exp((double)logits[i] - mraw);",
     "  for (int i = 0; i < V; ++i) zraw += exp((double)logits[i] - mraw + 0.25 * (i == 0));"),
    ("prefill attends one key too far", "const int n = pos[t] + 1; /* keys [0, pos] */",
     "const int n = pos[t] + 2; /* keys [0, pos] */"),
    ("prefill excludes the token itself", "const int n = pos[t] + 1; /* keys [0, pos] */",
     "const int n = pos[t] > 0 ? pos[t] : 1; /* keys [0, pos] */"),
    ("prefill positions counted from the prefix start", "      pos[qo_indptr[b] + i] = pos0 + i;",
     "      pos[qo_indptr[b] + i] = i;"),
    ("prefill tokens appended one slot late", "        const int64_t pos = (int64_t)pos0 + i;",
     "        const int64_t pos = (int64_t)pos0 + i + 1;"),
    ("prefill keys of another request", "      const int32_t pg = page_table[(int64_t)b * max_pages + j / page_size];\n      const int64_t off = cache_offset(num_pages, page_size, num_kv_heads, D, layer,\n                                       pg, 0, j % page_size, g);",
     "      const int32_t pg = page_table[(int64_t)(b > 0 ? b - 1 : b) * max_pages + j / page_size];\n      const int64_t off = cache_offset(num_pages, page_size, num_kv_heads, D, layer,\n                                       pg, 0, j % page_size, g);"),
    ("gumbel noise indexed by the sorted rank",
     "double sc = ord[r].x + pkvo_gumbel(seed, salt, id, step);",
     "double sc = ord[r].x + pkvo_gumbel(seed, salt, r, step);"),
    ("gumbel counter words swapped",
     "double sc = ord[r].x + pkvo_gumbel(seed, salt, id, step);",
     "double sc = ord[r].x + pkvo_gumbel(seed, salt, step, id);"),
    ("penalty window from the oldest token",
     "pen[n_pen++] = history[(int64_t)s * hist_cap + (len - 1 - i) % hist_cap];",
     "pen[n_pen++] = history[(int64_t)s * hist_cap + i % hist_cap];"),
]


def _pins():
    """(name, callable) of the pin checks, cheapest first."""
    return [
        ("philox", lambda: [TS.test_philox_matches_numpy_raw_words(k, c) for k, c in [
            ((12345, 7), (41, 3, 0, 0)), ((2**64 - 1, 2**63 + 5), (2**64 - 1, 2**64 - 1, 9, 0))]]),
        ("uniform", TS.test_uniform_uses_word0_and_is_strictly_inside_unit_interval),
        ("exact draw", lambda: [TS.test_sampled_token_is_the_gumbel_argmax_of_numpy_philox_noise(v)
                                for v in (6, 16)]),
        ("batched draw", TS.test_batched_and_frame_draws_use_the_slot_step_and_call_salt),
        ("append", TA.test_append_writes_exactly_the_slot_and_nothing_else),
        ("sdpa", lambda: [TA.test_attention_matches_torch_sdpa_fp64(*a)
                          for a in [(4, 64, True), (3, 128, True)]]),
        ("single token", TA.test_single_token_returns_its_value),
        ("identical keys", TA.test_identical_keys_give_mean_of_values),
        ("halves", TA.test_two_halves_merge_by_lse_to_the_whole),
        ("prefill append", TP.test_append_tokens_bytes),
        ("prefill first token", TP.test_first_token_of_an_empty_prefix_attends_only_to_itself),
        ("prefill running mean", TP.test_identical_keys_give_the_running_mean_of_the_values),
        ("prefill decode", TP.test_one_new_token_per_request_is_the_decode_oracle),
        ("prefill chunked", TP.test_chunked_prefill_equals_one_step),
        ("prefill sdpa", lambda: [TP.test_prefill_oracle_matches_torch_sdpa_with_a_causal_mask(n)
                                  for n in TP.CASES]),
        ("greedy", lambda: [TS.test_greedy_is_numpy_argmax(t) for t in (0.0, 1e-6)]),
        ("top-k/top-p argmax", TS.test_top_k_one_and_tiny_top_p_are_argmax_for_any_seed),
        ("boundary p", TS.test_top_p_boundary_prefix_exactly_p_drops_the_next_token),
        ("crossing", TS.test_top_p_keeps_the_crossing_token),
        ("top-k ties", TS.test_top_k_tie_at_the_cut_goes_to_lower_ids),
        ("kept sets", lambda: [TS.test_kept_set_count_matches_brute_force(v) for v in (5, 8)]),
        ("frame salts", TS.test_frame_without_feedback_equals_independent_salted_samples),
        ("frame feedback", TS.test_frame_feedback_wiring),
        ("full frame gating", TS.test_full_frame_channel0_is_the_salt0_sample_and_gates_the_codes),
        ("full frame never stops", TS.test_full_frame_that_never_stops_is_the_codebook_frame),
        ("full frame always stops", TS.test_full_frame_that_always_stops_is_a_pad_row),
        ("ext off", TS.test_ext_with_the_controls_off_is_the_base_sampler),
        ("raw logprob", TS.test_raw_logprob_is_scipy_log_softmax_of_the_unprocessed_logits),
        ("processed logprob forms", TS.test_processed_logprob_closed_forms),
        ("penalty rule", TS.test_repetition_penalty_rule_closed_form),
        ("min_p ties", TS.test_min_p_keeps_exactly_the_ties_with_the_maximum_at_one),
        ("history ring", TS.test_seeded_sample_ext_history_ring_and_window),
        ("processed logprob freq", lambda: TS.test_processed_logprob_is_the_sampling_distribution(
            0.8, 6, 0.9, 0.05, 1.8)),
        ("gumbel moments", TS.test_gumbel_moments),
        ("chi-square", lambda: TS.test_gumbel_max_frequencies_chi_square(0, 1.0, 1.0)),
    ]


def test_every_mutant_source_edit_applies_once():
    src = oracle.source_text()
    for name, old, _ in MUTANTS:
        assert src.count(old) == 1, name


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, workdir):
    src = oracle.source_text().replace(old, new)
    path = os.path.join(workdir, "mutant_%d.so" % abs(hash(name)))
    oracle.compile_variant(src, path)
    caught = None
    with oracle.using_library(path):
        for pin, fn in _pins():
            try:
                fn()
            except AssertionError:
                caught = pin
                break
    assert caught is not None, "no pin catches: %s" % name
