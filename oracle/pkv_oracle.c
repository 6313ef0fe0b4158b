/*
 * pkv_oracle.c -- plain fp64 CPU oracle for one batched decode step over a
 * paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file.  It is used by tests/, by __graft_entry__.smoke()
 * and by bench.py's cpu_baseline / reference arm, and nowhere else.  It
 * shares no code, header, table or helper with the CUDA library: the two are
 * written independently and only meet in the tests, on the same inputs.
 *
 * What it computes, step by step, in the order of the source pages:
 *
 *   kv_append      -- "Adding a Model" (vox-serve docs), section "1. The model
 *                     code": each layer writes its new keys and values into
 *                     the paged cache laid out
 *                     [num_layers, num_pages, 2, page_size, num_kv_heads,
 *                     head_dim]; section "How a program runs": padding
 *                     entries (active == 0) point at KV page 0 and must not
 *                     write into other requests' state.
 *   decode attn    -- same section: attention "through the paged KV cache";
 *                     grouped-query heads from num_qo_heads / num_kv_heads
 *                     (section "2. The program").  Written as gather, then a
 *                     plain softmax, then a weighted sum: no online softmax,
 *                     no splitting, no reordering.
 *   prefill        -- "Adding a Model", "How a program runs": lm_prefill
 *                     runs prompt rows (row buckets); "Supported Models",
 *                     Qwen3.5 / Qwen3.8 notes: text prefill and mixed
 *                     steps.  Each request's new tokens are appended at
 *                     consecutive positions ending at seq_len - 1 and each
 *                     attends causally to its request's positions up to
 *                     its own (a decode row is one new token).
 *   seeded sample  -- "Supported Models" (mstar docs), "Fish Audio S2-Pro
 *                     notes": temperature first, then top-k and top-p over the
 *                     tempered probabilities, and the top-p boundary keeps the
 *                     token that carries the running total past top-p;
 *                     "Chatterbox notes": temperature under 1e-5 is greedy
 *                     and a top-k of the whole vocabulary or more is no
 *                     filter; "Adding a Model", "How a program runs": draws
 *                     come from per-request seeds so that a request samples
 *                     the same tokens whatever batch it lands in, with a
 *                     different salt per sampling call (section "2. The
 *                     program", decode_tokens); stop_tokens() / audio_tokens()
 *                     classify the sampled token into out_kind.
 *   frame loop     -- MOSS-TTS-Local on SGLang-Omni (mosi.cn blog), section
 *                     on the model: per frame, one local-transformer layer
 *                     first gives a stop/continue decision, then 12 RVQ
 *                     codebooks are sampled in order, each fed back before
 *                     the next; a frame row holds 13 channels, channel 0
 *                     the control token and 1..12 the codes; section
 *                     "AR Engine": the 13 samplings of a frame run on a
 *                     seeded GPU sampler with per-request seeds and
 *                     counters.
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes of the repository):
 *   - dim 2 of the cache: index 0 holds K, index 1 holds V;
 *   - q head h uses kv head h / (num_qo_heads / num_kv_heads);
 *   - seq_len counts the token being appended; it is written at position
 *     seq_len - 1 and attention covers positions [0, seq_len);
 *   - softmax scale is an argument (1/sqrt(head_dim) by default);
 *   - padding rows: append writes page 0, slot 0; attention returns zeros
 *     and lse = -inf; the sampler returns token 0 of kind OTHER and leaves
 *     the per-slot step counter alone;
 *   - ordering is (value descending, token id ascending) everywhere;
 *   - top-k first (0 or >= V: off), then top-p over the top-k survivors
 *     renormalised: token r (in order) is kept iff r == 0 or
 *     S_{r-1} < p * Z, S the running sum of exp(x - x_max) in sorted order
 *     and Z the same sum over all top-k survivors;
 *   - randomness: Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel
 *     random numbers: as easy as 1, 2, 3", SC 2011), key = (seed, salt),
 *     counter = (token id, step, 0, 0); word 0 gives
 *     u = (2 * (w >> 12) + 1) * 2^-53, exactly representable and strictly
 *     inside (0, 1); Gumbel noise g = -log(-log(u)); the sample is the
 *     argmax over kept tokens of x + g (lowest id on exact ties);
 *   - frame loop feedback (no trained weights exist): the logits of
 *     codebook j > 0 are base[j] + fb[j][code_{j-1}], the add rounded once
 *     to fp32 like any fp32 logits tensor; salt = 1 + j; the per-slot step
 *     is read once per frame and advanced once per frame;
 *   - the stop/continue sample (no trained weights exist): channel 0
 *     samples caller-given control logits [B][Vc] with salt 0 and the
 *     slot's temperature / top-k / top-p; when it returns the caller's stop
 *     token, the frame's codebook channels hold the pad code -1, nothing
 *     else is sampled and the row's kind is STOP; otherwise the codebooks
 *     follow as above and the kind is AUDIO.  The control token does not
 *     feed the codebooks.
 *
 * Every floating-point decision here is taken in fp64 (bf16 and fp32 inputs
 * convert to double exactly).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define PKVO_KIND_OTHER 0
#define PKVO_KIND_AUDIO 1
#define PKVO_KIND_STOP 2
#define PKVO_CODE_PAD (-1) /* codebook channels of a frame that stopped */

/* ------------------------------------------------------------------ */
/* Number of threads OpenMP would use (1 without OpenMP).              */
/* ------------------------------------------------------------------ */
int pkvo_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void pkvo_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* bf16 -> double: the bf16 bits are the top half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Offset, in elements, of cache[layer][page][kv][slot][head][0]. */
static int64_t cache_offset(int64_t num_pages, int64_t page_size,
                            int64_t num_kv_heads, int64_t head_dim,
                            int64_t layer, int64_t page, int64_t kv,
                            int64_t slot, int64_t head) {
  int64_t off = layer;
  off = off * num_pages + page;
  off = off * 2 + kv;
  off = off * page_size + slot;
  off = off * num_kv_heads + head;
  return off * head_dim;
}

/* ------------------------------------------------------------------ */
/* KV append ("Adding a Model", section "1. The model code":           */
/* set_kv_cache writes each row's new k, v into its page slot).        */
/* Returns the number of active rows whose seq_len or page id is out   */
/* of range; those rows write nothing.                                  */
/* ------------------------------------------------------------------ */
int pkvo_kv_append(uint16_t *cache, int num_layers, int num_pages,
                   int page_size, int num_kv_heads, int head_dim, int layer,
                   const uint16_t *k, const uint16_t *v,
                   const int32_t *page_table, int max_pages,
                   const int32_t *seq_lens, const int32_t *active, int B) {
  (void)num_layers;
  int bad = 0;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  for (int b = 0; b < B; ++b) {
    int64_t page, slot;
    if (!active[b]) {
      /* padding entry: the dummy page 0, slot 0 */
      page = 0;
      slot = 0;
    } else {
      int32_t n = seq_lens[b];
      if (n < 1 || (int64_t)n > (int64_t)max_pages * page_size) {
        ++bad;
        continue;
      }
      int64_t pos = (int64_t)n - 1;
      page = page_table[(int64_t)b * max_pages + pos / page_size];
      slot = pos % page_size;
      if (page < 0 || page >= num_pages) {
        ++bad;
        continue;
      }
    }
    for (int kv = 0; kv < 2; ++kv) {
      const uint16_t *src = (kv == 0 ? k : v) + (int64_t)b * row;
      int64_t dst = cache_offset(num_pages, page_size, num_kv_heads, head_dim,
                                 layer, page, kv, slot, 0);
      memcpy(cache + dst, src, (size_t)row * sizeof(uint16_t));
    }
  }
  return bad;
}

/* ------------------------------------------------------------------ */
/* Paged decode attention ("Adding a Model", section "1. The model     */
/* code": attn_wrapper.run(q, kv_cache) over the paged layout; q head h */
/* reads kv head h / (Hq / Hkv)).                                       */
/*   q    bf16 [B][Hq][D]                                               */
/*   out  fp64 [B][Hq][D]   (zeros for padding rows)                    */
/*   lse  fp64 [B][Hq]      natural-log log-sum-exp of the scaled       */
/*                          scores (-inf for padding rows); may be NULL */
/* Returns the number of active rows with an out-of-range seq_len or   */
/* page id (their outputs are zeros).                                   */
/* ------------------------------------------------------------------ */
int pkvo_paged_decode_attn(const uint16_t *cache, int num_layers,
                           int num_pages, int page_size, int num_kv_heads,
                           int head_dim, int layer, const uint16_t *q,
                           int num_qo_heads, double sm_scale,
                           const int32_t *page_table, int max_pages,
                           const int32_t *seq_lens, const int32_t *active,
                           int B, double *out, double *lse) {
  (void)num_layers;
  const int D = head_dim;
  const int Hq = num_qo_heads;
  const int group = num_qo_heads / num_kv_heads;
  int bad = 0;

  /* Validate rows first (sequentially) so the parallel loop below does
   * no bookkeeping. */
  char *ok = (char *)calloc((size_t)(B > 0 ? B : 1), 1);
  for (int b = 0; b < B; ++b) {
    if (!active[b]) continue;
    int32_t n = seq_lens[b];
    int row_ok = (n >= 1 && (int64_t)n <= (int64_t)max_pages * page_size);
    if (row_ok) {
      int npages = (n + page_size - 1) / page_size;
      for (int i = 0; i < npages; ++i) {
        int32_t pg = page_table[(int64_t)b * max_pages + i];
        if (pg < 0 || pg >= num_pages) row_ok = 0;
      }
    }
    ok[b] = (char)row_ok;
    if (!row_ok) ++bad;
  }

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
    const int b = (int)(bh / Hq);
    const int h = (int)(bh % Hq);
    double *o = out + bh * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (lse) lse[bh] = -INFINITY;
    if (!active[b] || !ok[b]) continue;

    const int n = seq_lens[b];
    const int g = h / group;
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    for (int d = 0; d < D; ++d)
      qd[d] = bf16_bits_to_double(q[bh * D + d]);

    /* gather every key of the row through the page table; scores */
    for (int t = 0; t < n; ++t) {
      int32_t pg = page_table[(int64_t)b * max_pages + t / page_size];
      int64_t off = cache_offset(num_pages, page_size, num_kv_heads, D, layer,
                                 pg, 0, t % page_size, g);
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qd[d] * bf16_bits_to_double(cache[off + d]);
      s[t] = sm_scale * dot;
    }
    /* softmax */
    double m = s[0];
    for (int t = 1; t < n; ++t)
      if (s[t] > m) m = s[t];
    double z = 0.0;
    for (int t = 0; t < n; ++t) {
      s[t] = exp(s[t] - m);
      z += s[t];
    }
    /* weighted sum of the values */
    for (int t = 0; t < n; ++t) {
      int32_t pg = page_table[(int64_t)b * max_pages + t / page_size];
      int64_t off = cache_offset(num_pages, page_size, num_kv_heads, D, layer,
                                 pg, 1, t % page_size, g);
      double p = s[t] / z;
      for (int d = 0; d < D; ++d) o[d] += p * bf16_bits_to_double(cache[off + d]);
    }
    if (lse) lse[bh] = m + log(z);
    free(s);
    free(qd);
  }
  free(ok);
  return bad;
}

/* ------------------------------------------------------------------ */
/* Prefill / mixed steps ("Adding a Model", section "How a program     */
/* runs": lm_prefill feeds prompt rows, one graph per row bucket;       */
/* "Supported Models", Qwen3.5 / Qwen3.8 notes: text prefill and mixed  */
/* steps, a mixed step carrying decode rows beside prompt rows).        */
/* Request b brings q_b = qo_indptr[b+1] - qo_indptr[b] new tokens,     */
/* packed at rows [qo_indptr[b], qo_indptr[b+1]) of k, v and q; with    */
/* n_b = seq_lens[b] (counting them), token i sits at position          */
/* n_b - q_b + i.  A decode row is q_b = 1.  Padding requests           */
/* (active == 0) write every token to page 0, slot 0 and read nothing. */
/* ------------------------------------------------------------------ */

/* Request b's new tokens and their first position; 0 when the request
 * is malformed (q < 0, n < q, n < 1 with q > 0, n beyond the table, or
 * a page id out of range for one of its positions). */
static int prefill_request_ok(const int32_t *qo_indptr, const int32_t *page_table,
                              int max_pages, int page_size, int num_pages,
                              const int32_t *seq_lens, int b, int *q_out,
                              int *pos0_out) {
  const int q = qo_indptr[b + 1] - qo_indptr[b];
  const int n = seq_lens[b];
  *q_out = q;
  *pos0_out = n - q;
  if (q < 0 || n < q || (int64_t)n > (int64_t)max_pages * page_size) return 0;
  if (q > 0 && n < 1) return 0;
  const int npages = (n + page_size - 1) / page_size;
  for (int i = 0; i < npages; ++i) {
    const int32_t pg = page_table[(int64_t)b * max_pages + i];
    if (pg < 0 || pg >= num_pages) return 0;
  }
  return 1;
}

/* Multi-token append: token i of request b into the slot of position
 * n_b - q_b + i.  k, v bf16 [T][Hkv][D] with T = qo_indptr[B].  Returns
 * the number of malformed active requests (they write nothing). */
int pkvo_kv_append_tokens(uint16_t *cache, int num_layers, int num_pages,
                          int page_size, int num_kv_heads, int head_dim,
                          int layer, const uint16_t *k, const uint16_t *v,
                          const int32_t *qo_indptr, const int32_t *page_table,
                          int max_pages, const int32_t *seq_lens,
                          const int32_t *active, int B) {
  (void)num_layers;
  int bad = 0;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  for (int b = 0; b < B; ++b) {
    int q, pos0;
    const int ok = prefill_request_ok(qo_indptr, page_table, max_pages, page_size,
                                      num_pages, seq_lens, b, &q, &pos0);
    if (active[b] && !ok) {
      ++bad;
      continue;
    }
    if (!active[b] && q < 0) continue;
    for (int i = 0; i < q; ++i) {
      int64_t page = 0, slot = 0; /* padding: the dummy page 0, slot 0 */
      if (active[b]) {
        const int64_t pos = (int64_t)pos0 + i;
        page = page_table[(int64_t)b * max_pages + pos / page_size];
        slot = pos % page_size;
      }
      const int64_t t = (int64_t)qo_indptr[b] + i;
      for (int kv = 0; kv < 2; ++kv) {
        const uint16_t *src = (kv == 0 ? k : v) + t * row;
        const int64_t dst = cache_offset(num_pages, page_size, num_kv_heads, head_dim,
                                         layer, page, kv, slot, 0);
        memcpy(cache + dst, src, (size_t)row * sizeof(uint16_t));
      }
    }
  }
  return bad;
}

/* Causal attention of the new tokens over the paged cache: the token at
 * position p attends to positions [0, p] of its own request (what was
 * cached before the step and the step's tokens up to itself), with the
 * same gather / plain softmax / weighted sum as the decode oracle.
 *   q    bf16 [T][Hq][D];  out fp64 [T][Hq][D];  lse fp64 [T][Hq] or NULL.
 * Rows of padding or malformed requests get zeros and lse = -inf.
 * Returns the number of malformed active requests. */
int pkvo_prefill_attn(const uint16_t *cache, int num_layers, int num_pages,
                      int page_size, int num_kv_heads, int head_dim, int layer,
                      const uint16_t *q, int num_qo_heads, double sm_scale,
                      const int32_t *qo_indptr, const int32_t *page_table,
                      int max_pages, const int32_t *seq_lens,
                      const int32_t *active, int B, double *out, double *lse) {
  (void)num_layers;
  const int D = head_dim;
  const int Hq = num_qo_heads;
  const int group = num_qo_heads / num_kv_heads;
  const int64_t T = qo_indptr[B];
  int bad = 0;
  /* owner request, position and validity of every token row */
  int32_t *req = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
  int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
  for (int64_t t = 0; t < T; ++t) req[t] = -1;
  for (int b = 0; b < B; ++b) {
    int qn, pos0;
    const int ok = prefill_request_ok(qo_indptr, page_table, max_pages, page_size,
                                      num_pages, seq_lens, b, &qn, &pos0);
    if (active[b] && !ok) ++bad;
    if (!active[b] || !ok) continue;
    for (int i = 0; i < qn; ++i) {
      req[qo_indptr[b] + i] = b;
      pos[qo_indptr[b] + i] = pos0 + i;
    }
  }

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t th = 0; th < T * Hq; ++th) {
    const int64_t t = th / Hq;
    const int h = (int)(th % Hq);
    double *o = out + th * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (lse) lse[th] = -INFINITY;
    const int b = req[t];
    if (b < 0) continue;
    const int n = pos[t] + 1; /* keys [0, pos] */
    const int g = h / group;
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    for (int d = 0; d < D; ++d) qd[d] = bf16_bits_to_double(q[th * D + d]);
    for (int j = 0; j < n; ++j) {
      const int32_t pg = page_table[(int64_t)b * max_pages + j / page_size];
      const int64_t off = cache_offset(num_pages, page_size, num_kv_heads, D, layer,
                                       pg, 0, j % page_size, g);
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qd[d] * bf16_bits_to_double(cache[off + d]);
      s[j] = sm_scale * dot;
    }
    double m = s[0];
    for (int j = 1; j < n; ++j)
      if (s[j] > m) m = s[j];
    double z = 0.0;
    for (int j = 0; j < n; ++j) {
      s[j] = exp(s[j] - m);
      z += s[j];
    }
    for (int j = 0; j < n; ++j) {
      const int32_t pg = page_table[(int64_t)b * max_pages + j / page_size];
      const int64_t off = cache_offset(num_pages, page_size, num_kv_heads, D, layer,
                                       pg, 1, j % page_size, g);
      const double p = s[j] / z;
      for (int d = 0; d < D; ++d) o[d] += p * bf16_bits_to_double(cache[off + d]);
    }
    if (lse) lse[th] = m + log(z);
    free(s);
    free(qd);
  }
  free(pos);
  free(req);
  return bad;
}

/* ------------------------------------------------------------------ */
/* Philox4x64-10, from the definition in Salmon et al., SC 2011:       */
/* a 4-word counter is mixed by 10 rounds; each round multiplies two   */
/* words by fixed odd constants, keeps the high and low halves of the  */
/* 128-bit products, and xors the high halves with the other two words */
/* and the round key; the round key is bumped by two Weyl constants    */
/* between rounds.                                                      */
/* ------------------------------------------------------------------ */
static const uint64_t PHILOX_M0 = 0xD2E7470EE14C6C93ULL;
static const uint64_t PHILOX_M1 = 0xCA5A826395121157ULL;
static const uint64_t PHILOX_W0 = 0x9E3779B97F4A7C15ULL; /* golden ratio */
static const uint64_t PHILOX_W1 = 0xBB67AE8584CAA73BULL; /* sqrt(3) - 1 */

void pkvo_philox4x64_10(const uint64_t key_in[2], const uint64_t ctr_in[4],
                        uint64_t out[4]) {
  uint64_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
  uint64_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    unsigned __int128 p0 = (unsigned __int128)PHILOX_M0 * x0;
    unsigned __int128 p1 = (unsigned __int128)PHILOX_M1 * x2;
    uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
    uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
    uint64_t y0 = hi1 ^ x1 ^ k0;
    uint64_t y1 = lo1;
    uint64_t y2 = hi0 ^ x3 ^ k1;
    uint64_t y3 = lo0;
    x0 = y0;
    x1 = y1;
    x2 = y2;
    x3 = y3;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

/* The uniform of token `token` at step `step` of the stream (seed, salt). */
double pkvo_uniform(uint64_t seed, uint32_t salt, int64_t token, int64_t step) {
  uint64_t key[2] = {seed, (uint64_t)salt};
  uint64_t ctr[4] = {(uint64_t)token, (uint64_t)step, 0, 0};
  uint64_t w[4];
  pkvo_philox4x64_10(key, ctr, w);
  uint64_t j = w[0] >> 12; /* 52 random bits */
  return (double)(2 * j + 1) * 0x1p-53;
}

double pkvo_gumbel(uint64_t seed, uint32_t salt, int64_t token, int64_t step) {
  double u = pkvo_uniform(seed, salt, token, step);
  return -log(-log(u));
}

/* ------------------------------------------------------------------ */
/* Seeded temperature / top-k / top-p sampling of one row.             */
/* ------------------------------------------------------------------ */
typedef struct {
  int32_t token;
  int32_t n_kept;       /* tokens that survived top-k and top-p */
  int32_t greedy;       /* 1 when temperature <= 1e-5 */
  int32_t pad_;
  double top2_gap_rel;  /* (best - second) / max(1, |best|) over kept, +inf if 1 kept */
  double member_margin; /* min distance of a top-p prefix sum from p*Z, relative to Z,
                           and of exp(x - x_max) from min_p at the min_p cut
                           (+inf when both are off or no boundary exists) */
  double logprob_raw;   /* log-softmax of the unprocessed logits at the token */
  double logprob_proc;  /* log-probability of the token in the distribution it
                           was drawn from (0 for greedy) */
} pkvo_sample_info;

typedef struct {
  double x;
  int32_t id;
} xid_t;

/* (x descending, id ascending) */
static int cmp_xid(const void *a, const void *b) {
  const xid_t *p = (const xid_t *)a, *q = (const xid_t *)b;
  if (p->x > q->x) return -1;
  if (p->x < q->x) return 1;
  return (p->id > q->id) - (p->id < q->id);
}

/* logits: fp32 [V].  Returns the sampled token.  The order of the
 * transforms is the pages' (Chatterbox notes: repetition penalty ->
 * temperature -> min_p -> top_p), with top-k after the temperature:
 *   1. repetition penalty: each distinct id of pen_tokens[0..n_pen) in
 *      [0, V) gets logit / rep_penalty if the logit is positive, else
 *      logit * rep_penalty, in fp32 like the logits (rep_penalty 1: off);
 *   2. temperature: x = logit / T (<= 1e-5: greedy argmax, lowest id);
 *   3. top-k (0 or >= V: off);
 *   4. min_p (<= 0: off): rank r of the order is kept iff r == 0 or
 *      exp(x_r - x_max) >= min_p;
 *   5. top-p over the renormalised survivors (R7 rule);
 *   6. Gumbel-max over the kept tokens.
 * info (may be NULL) also gets the log-softmax of the raw logits at the
 * token and its log-probability under the renormalised kept set. */
int32_t pkvo_sample_row_ext(const float *logits, int V, uint64_t seed, int64_t step,
                            uint32_t salt, float temperature, int32_t top_k,
                            float top_p, float min_p, float rep_penalty,
                            const int32_t *pen_tokens, int n_pen,
                            pkvo_sample_info *info) {
  pkvo_sample_info local;
  if (!info) info = &local;
  memset(info, 0, sizeof *info);
  info->top2_gap_rel = INFINITY;
  info->member_margin = INFINITY;

  /* raw log-softmax normaliser */
  double mraw = -INFINITY, zraw = 0.0;
  for (int i = 0; i < V; ++i)
    if ((double)logits[i] > mraw) mraw = (double)logits[i];
  for (int i = 0; i < V; ++i) zraw += exp((double)logits[i] - mraw);
  const double lse_raw = mraw + log(zraw);

  /* 1. repetition penalty on a copy */
  float *pl = (float *)malloc(sizeof(float) * (size_t)(V > 0 ? V : 1));
  memcpy(pl, logits, sizeof(float) * (size_t)V);
  if (rep_penalty != 1.0f && n_pen > 0) {
    unsigned char *done = (unsigned char *)calloc((size_t)V, 1);
    for (int i = 0; i < n_pen; ++i) {
      const int32_t t = pen_tokens[i];
      if (t < 0 || t >= V || done[t]) continue;
      done[t] = 1;
      pl[t] = pl[t] > 0.0f ? pl[t] / rep_penalty : pl[t] * rep_penalty;
    }
    free(done);
  }

  if (!(temperature > 1e-5f)) {
    /* greedy: the first maximum, i.e. the lowest id among equal logits */
    int32_t best = 0;
    for (int i = 1; i < V; ++i)
      if (pl[i] > pl[best]) best = i;
    info->token = best;
    info->n_kept = 1;
    info->greedy = 1;
    info->logprob_raw = (double)logits[best] - lse_raw;
    info->logprob_proc = 0.0;
    free(pl);
    return best;
  }

  xid_t *ord = (xid_t *)malloc(sizeof(xid_t) * (size_t)V);
  const double T = (double)temperature;
  for (int i = 0; i < V; ++i) {
    ord[i].x = (double)pl[i] / T;
    ord[i].id = i;
  }
  qsort(ord, (size_t)V, sizeof(xid_t), cmp_xid);

  /* top-k: 0 or >= V means no filter */
  int K = (top_k > 0 && top_k < V) ? top_k : V;

  const double m = ord[0].x;
  double *e = (double *)malloc(sizeof(double) * (size_t)K);
  for (int r = 0; r < K; ++r) e[r] = exp(ord[r].x - m);

  /* min_p over the top-k survivors */
  int Kp = K;
  if (min_p > 0.0f) {
    Kp = 1;
    while (Kp < K && e[Kp] >= (double)min_p) ++Kp;
    double d = fabs(e[Kp - 1] - (double)min_p);
    if (Kp < K && fabs(e[Kp] - (double)min_p) < d) d = fabs(e[Kp] - (double)min_p);
    if (Kp > 1 || Kp < K) info->member_margin = d;
  }

  /* top-p over the renormalised survivors */
  int kept = Kp;
  double S = 0.0; /* mass of the kept tokens */
  for (int r = 0; r < Kp; ++r) S += e[r];
  if (top_p < 1.0f) {
    const double Z = S;
    const double pz = (double)top_p * Z;
    S = 0.0; /* S_{r-1}: mass of the tokens before r */
    kept = 0;
    for (int r = 0; r < Kp; ++r) {
      if (r == 0 || S < pz) {
        kept = r + 1;
        S += e[r];
      } else {
        break;
      }
    }
    /* near-tie diagnostics: how close the two prefix sums around the cut
       lie to p*Z */
    {
      double Sprev = 0.0; /* S before the last kept token */
      for (int r = 0; r + 1 < kept; ++r) Sprev += e[r];
      double margin = INFINITY;
      if (kept >= 2) margin = fabs(pz - Sprev) / Z;
      if (kept < Kp) {
        double d2 = fabs(S - pz) / Z;
        if (d2 < margin) margin = d2;
      }
      if (margin < info->member_margin) info->member_margin = margin;
    }
  }

  /* Gumbel-max over the kept tokens */
  double best = -INFINITY, second = -INFINITY;
  int32_t best_id = ord[0].id;
  double best_x = ord[0].x;
  for (int r = 0; r < kept; ++r) {
    int32_t id = ord[r].id;
    double sc = ord[r].x + pkvo_gumbel(seed, salt, id, step);
    if (sc > best || (sc == best && id < best_id)) {
      second = best;
      best = sc;
      best_id = id;
      best_x = ord[r].x;
    } else if (sc > second) {
      second = sc;
    }
  }
  if (kept >= 2) {
    double scale = fabs(best) > 1.0 ? fabs(best) : 1.0;
    info->top2_gap_rel = (best - second) / scale;
  }
  info->token = best_id;
  info->n_kept = kept;
  info->logprob_raw = (double)logits[best_id] - lse_raw;
  info->logprob_proc = (best_x - m) - log(S);
  free(e);
  free(ord);
  free(pl);
  return best_id;
}

int32_t pkvo_sample_row(const float *logits, int V, uint64_t seed, int64_t step,
                        uint32_t salt, float temperature, int32_t top_k,
                        float top_p, pkvo_sample_info *info) {
  return pkvo_sample_row_ext(logits, V, seed, step, salt, temperature, top_k, top_p, 0.0f,
                             1.0f, NULL, 0, info);
}

/* stop_tokens() / audio_tokens() of "Adding a Model", section "2. The
 * program": STOP if the token is a stop token, else AUDIO inside
 * [audio_lo, audio_hi), else OTHER. */
int32_t pkvo_token_kind(int32_t tok, const int32_t *stop_tokens, int n_stop,
                        int32_t audio_lo, int32_t audio_hi) {
  for (int i = 0; i < n_stop; ++i)
    if (stop_tokens[i] == tok) return PKVO_KIND_STOP;
  if (tok >= audio_lo && tok < audio_hi) return PKVO_KIND_AUDIO;
  return PKVO_KIND_OTHER;
}

/* ------------------------------------------------------------------ */
/* Batched seeded sampling: rows in, out_tok / out_kind out.           */
/* logits fp32 [B][row_stride]; per-slot state indexed by slots[b].    */
/* Padding rows (active == 0) give token 0, kind OTHER, and leave the  */
/* step counters alone.  Returns the number of active rows whose slot  */
/* is out of range (they give token 0, kind OTHER).                     */
/* info may be NULL; else it receives one record per row.               */
/* ------------------------------------------------------------------ */
int pkvo_seeded_sample(const float *logits, int64_t row_stride, int B, int V,
                       const int32_t *slots, const int32_t *active,
                       int num_slots, const uint64_t *seeds, int64_t *steps,
                       const float *temperature, const int32_t *top_k,
                       const float *top_p, uint32_t salt, int advance,
                       const int32_t *stop_tokens, int n_stop,
                       int32_t audio_lo, int32_t audio_hi, int32_t *out_tok,
                       int32_t *out_kind, pkvo_sample_info *info) {
  int bad = 0;
  for (int b = 0; b < B; ++b) {
    if (info) {
      memset(&info[b], 0, sizeof info[b]);
      info[b].top2_gap_rel = INFINITY;
      info[b].member_margin = INFINITY;
    }
    out_tok[b] = 0;
    out_kind[b] = PKVO_KIND_OTHER;
    if (!active[b]) continue;
    int32_t s = slots[b];
    if (s < 0 || s >= num_slots) {
      ++bad;
      continue;
    }
    int32_t tok = pkvo_sample_row(logits + (int64_t)b * row_stride, V, seeds[s],
                                  steps[s], salt, temperature[s], top_k[s],
                                  top_p[s], info ? &info[b] : NULL);
    out_tok[b] = tok;
    out_kind[b] = pkvo_token_kind(tok, stop_tokens, n_stop, audio_lo, audio_hi);
  }
  if (advance) {
    for (int b = 0; b < B; ++b) {
      if (!active[b]) continue;
      int32_t s = slots[b];
      if (s < 0 || s >= num_slots) continue;
      steps[s] += 1;
    }
  }
  return bad;
}

/* ------------------------------------------------------------------ */
/* pkvo_seeded_sample with the further sampling controls of the        */
/* program's sampler settings ("Adding a Model", section "2. The       */
/* program": min_p, repetition_penalty, repetition_window) in the      */
/* order of pkvo_sample_row_ext, and the raw / processed log-probs     */
/* ("Adding a Model": enable_logprobs, "logprobs_mode": "processed").   */
/*   min_p, rep_penalty float [num_slots], rep_window int32 [num_slots] */
/*   (each may be NULL: off / off / whole history);                    */
/*   history int32 [num_slots][hist_cap], hist_len int32 [num_slots]:  */
/*   the slot's sampled tokens as a ring (token n at n % hist_cap);     */
/*   the penalised ids are the last w = min(window, hist_len, hist_cap) */
/*   (window < 0: min(hist_len, hist_cap); 0: none) of them.  With      */
/*   advance, the sampled token is appended (history may be NULL: no   */
/*   penalty and nothing appended).  logprob_raw / logprob_proc float  */
/*   [B] (each may be NULL); padding rows get 0.                       */
/* ------------------------------------------------------------------ */
int pkvo_seeded_sample_ext(const float *logits, int64_t row_stride, int B, int V,
                           const int32_t *slots, const int32_t *active,
                           int num_slots, const uint64_t *seeds, int64_t *steps,
                           const float *temperature, const int32_t *top_k,
                           const float *top_p, const float *min_p,
                           const float *rep_penalty, const int32_t *rep_window,
                           int32_t *history, int32_t *hist_len, int hist_cap,
                           uint32_t salt, int advance, int32_t *out_tok,
                           float *logprob_raw, float *logprob_proc,
                           pkvo_sample_info *info) {
  int bad = 0;
  int32_t *pen = (int32_t *)malloc(sizeof(int32_t) * (size_t)(hist_cap > 0 ? hist_cap : 1));
  for (int b = 0; b < B; ++b) {
    pkvo_sample_info local;
    pkvo_sample_info *in = info ? &info[b] : &local;
    memset(in, 0, sizeof *in);
    in->top2_gap_rel = INFINITY;
    in->member_margin = INFINITY;
    out_tok[b] = 0;
    if (logprob_raw) logprob_raw[b] = 0.0f;
    if (logprob_proc) logprob_proc[b] = 0.0f;
    if (!active[b]) continue;
    int32_t s = slots[b];
    if (s < 0 || s >= num_slots) {
      ++bad;
      continue;
    }
    int n_pen = 0;
    if (history && hist_cap > 0) {
      const int64_t len = hist_len[s];
      const int32_t w = rep_window ? rep_window[s] : -1;
      int64_t n = len < hist_cap ? len : hist_cap;
      if (w >= 0 && w < n) n = w;
      for (int64_t i = 0; i < n; ++i) pen[n_pen++] = history[(int64_t)s * hist_cap + (len - 1 - i) % hist_cap];
    }
    int32_t tok = pkvo_sample_row_ext(logits + (int64_t)b * row_stride, V, seeds[s], steps[s],
                                      salt, temperature[s], top_k[s], top_p[s],
                                      min_p ? min_p[s] : 0.0f,
                                      rep_penalty ? rep_penalty[s] : 1.0f, pen, n_pen, in);
    out_tok[b] = tok;
    if (logprob_raw) logprob_raw[b] = (float)in->logprob_raw;
    if (logprob_proc) logprob_proc[b] = (float)in->logprob_proc;
  }
  free(pen);
  if (advance) {
    for (int b = 0; b < B; ++b) {
      if (!active[b]) continue;
      int32_t s = slots[b];
      if (s < 0 || s >= num_slots) continue;
      steps[s] += 1;
      if (history && hist_cap > 0) {
        history[(int64_t)s * hist_cap + hist_len[s] % hist_cap] = out_tok[b];
        hist_len[s] += 1;
      }
    }
  }
  return bad;
}

/* ------------------------------------------------------------------ */
/* The frame-local codebook loop (MOSS-TTS-Local blog: per frame, the  */
/* RVQ codebooks are sampled in order, each fed back before the next). */
/*   base fp32 [n_cb][B][V]; fb fp32 [n_cb][V][V] or NULL;            */
/*   out_codes int32 [B][n_cb]; out_kind int32 [B].                    */
/* Codebook j samples with salt 1 + j at the frame's step; the step is */
/* advanced once per frame for each active row.  Returns the number of */
/* active rows whose slot is out of range.  info may be NULL, else it  */
/* receives [B][n_cb] records.                                          */
/* ------------------------------------------------------------------ */
/* The codebooks of row b in order at the given step: codebook j samples
 * base[j][b] (+ fb[j][code_{j-1}] for j > 0) with salt 1 + j.  Writes
 * codes[j] and, when info is not NULL, info[j].  row: scratch of V floats. */
static void frame_codes_row(const float *base, const float *fb, int n_cb, int B,
                            int V, int b, uint64_t seed, int64_t step,
                            float temperature, int32_t top_k, float top_p,
                            float *row, int32_t *codes,
                            pkvo_sample_info *info) {
  int32_t prev = 0;
  for (int j = 0; j < n_cb; ++j) {
    const float *bj = base + ((int64_t)j * B + b) * V;
    if (j > 0 && fb) {
      const float *fj = fb + ((int64_t)j * V + prev) * V;
      /* The fp32 sum, rounded once: the exact sum of two binary32 values
       * rounded to binary64 and then to binary32 equals the binary32
       * rounding of the exact sum, since 53 >= 2 * 24 + 2. */
      for (int i = 0; i < V; ++i) row[i] = (float)((double)bj[i] + (double)fj[i]);
    } else {
      for (int i = 0; i < V; ++i) row[i] = bj[i];
    }
    prev = pkvo_sample_row(row, V, seed, step, (uint32_t)(1 + j), temperature,
                           top_k, top_p, info ? &info[j] : NULL);
    codes[j] = prev;
  }
}

static void clear_info(pkvo_sample_info *r) {
  memset(r, 0, sizeof *r);
  r->top2_gap_rel = INFINITY;
  r->member_margin = INFINITY;
}

int pkvo_codebook_frame_sample(const float *base, const float *fb, int n_cb,
                               int B, int V, const int32_t *slots,
                               const int32_t *active, int num_slots,
                               const uint64_t *seeds, int64_t *steps,
                               const float *temperature, const int32_t *top_k,
                               const float *top_p, int32_t *out_codes,
                               int32_t *out_kind, pkvo_sample_info *info) {
  int bad = 0;
  float *row = (float *)malloc(sizeof(float) * (size_t)(V > 0 ? V : 1));
  for (int b = 0; b < B; ++b) {
    for (int j = 0; j < n_cb; ++j) {
      out_codes[(int64_t)b * n_cb + j] = 0;
      if (info) clear_info(&info[(int64_t)b * n_cb + j]);
    }
    out_kind[b] = PKVO_KIND_OTHER;
    if (!active[b]) continue;
    int32_t s = slots[b];
    if (s < 0 || s >= num_slots) {
      ++bad;
      continue;
    }
    frame_codes_row(base, fb, n_cb, B, V, b, seeds[s], steps[s], temperature[s],
                    top_k[s], top_p[s], row, out_codes + (int64_t)b * n_cb,
                    info ? &info[(int64_t)b * n_cb] : NULL);
    out_kind[b] = PKVO_KIND_AUDIO;
  }
  for (int b = 0; b < B; ++b) {
    if (!active[b]) continue;
    int32_t s = slots[b];
    if (s < 0 || s >= num_slots) continue;
    steps[s] += 1;
  }
  free(row);
  return bad;
}

/* ------------------------------------------------------------------ */
/* A full frame row: the stop/continue sample on channel 0, then the   */
/* codebooks (MOSS-TTS-Local blog, section on the model: 13 channels,  */
/* a stop/continue decision first, then the 12 codebooks in order).    */
/*   ctrl fp32 [B][Vc]; base, fb as above;                             */
/*   out_rows int32 [B][1 + n_cb]; out_kind int32 [B].                  */
/* Channel 0 samples ctrl[b] with salt 0 at the frame's step; when it   */
/* returns stop_ctrl, channels 1..n_cb hold PKVO_CODE_PAD and the kind  */
/* is STOP, else they hold the codes and the kind is AUDIO.  The step   */
/* is advanced once per frame for each active row.  Padding rows (and  */
/* rows whose slot is out of range) get zeros and OTHER.  info may be   */
/* NULL, else it receives [B][1 + n_cb] records (channel order).        */
/* Returns the number of active rows whose slot is out of range.        */
/* ------------------------------------------------------------------ */
int pkvo_frame_sample(const float *ctrl, int Vc, int32_t stop_ctrl,
                      const float *base, const float *fb, int n_cb, int B, int V,
                      const int32_t *slots, const int32_t *active, int num_slots,
                      const uint64_t *seeds, int64_t *steps,
                      const float *temperature, const int32_t *top_k,
                      const float *top_p, int32_t *out_rows, int32_t *out_kind,
                      pkvo_sample_info *info) {
  const int W = 1 + n_cb;
  int bad = 0;
  float *row = (float *)malloc(sizeof(float) * (size_t)(V > 0 ? V : 1));
  for (int b = 0; b < B; ++b) {
    int32_t *r = out_rows + (int64_t)b * W;
    for (int j = 0; j < W; ++j) {
      r[j] = 0;
      if (info) clear_info(&info[(int64_t)b * W + j]);
    }
    out_kind[b] = PKVO_KIND_OTHER;
    if (!active[b]) continue;
    int32_t s = slots[b];
    if (s < 0 || s >= num_slots) {
      ++bad;
      continue;
    }
    r[0] = pkvo_sample_row(ctrl + (int64_t)b * Vc, Vc, seeds[s], steps[s], 0u,
                           temperature[s], top_k[s], top_p[s],
                           info ? &info[(int64_t)b * W] : NULL);
    if (r[0] == stop_ctrl) {
      for (int j = 1; j < W; ++j) r[j] = PKVO_CODE_PAD;
      out_kind[b] = PKVO_KIND_STOP;
      continue;
    }
    frame_codes_row(base, fb, n_cb, B, V, b, seeds[s], steps[s], temperature[s],
                    top_k[s], top_p[s], row, r + 1,
                    info ? &info[(int64_t)b * W + 1] : NULL);
    out_kind[b] = PKVO_KIND_AUDIO;
  }
  for (int b = 0; b < B; ++b) {
    if (!active[b]) continue;
    int32_t s = slots[b];
    if (s < 0 || s >= num_slots) continue;
    steps[s] += 1;
  }
  free(row);
  return bad;
}
