/*
 * pkv.h -- C ABI of the GB300 (sm_103a) paged-KV decode step.
 *
 * One batched decode step over a paged KV cache, as the vox-serve docs
 * ("Adding a Model") state the problem: rows in; out_tok / out_kind out;
 * padding entries (active == 0) point at a dummy slot and KV page 0, do
 * real (ignored) work and never write another request's state; a request
 * samples the same tokens whatever batch it lands in.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All array pointers are DEVICE pointers owned by the caller.  The
 *    library allocates nothing, frees nothing, never synchronises and never
 *    reads device memory from the host.
 *  - `stream` is a cudaStream_t (NULL: the legacy default stream).  Work is
 *    stream-ordered; launch shapes depend only on the scalar arguments, so a
 *    call may be captured into a CUDA graph and replayed.
 *  - Return value: PKV_OK, or an error status.  Host-side argument errors are
 *    reported before anything is launched.  PKV_ERR_CUDA reports a launch
 *    error (cudaGetLastError, which does not synchronise).
 *  - Data errors found on the device (a page id outside [0, num_pages), a
 *    seq_len outside [1, max_pages * page_size], a slot outside
 *    [0, num_slots), a non-finite logit) are never trapped: the kernel
 *    avoids the bad access (page 0 / slot 0 / no write instead), ORs a
 *    PKV_DEV_ERR_* bit into *err_word when err_word is not NULL, and the
 *    affected row's outputs are unspecified.  Other rows are unaffected.
 *  - Page 0 and slot 0 are reserved for padding entries; no request may own
 *    them.  Slots of the active rows of one call must be distinct.
 *  - Tensors are C-contiguous unless a stride argument says otherwise.
 *    The cache, k, v and q must be 16-byte aligned; fp32 logits 4-byte.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define PKV_OK 0
#define PKV_ERR_INVALID_ARG 1 /* null pointer, non-positive size, bad shape */
#define PKV_ERR_UNSUPPORTED 2 /* valid, but outside what the kernels cover   */
#define PKV_ERR_CUDA 3        /* a kernel launch failed                       */
#define PKV_ERR_WORKSPACE 4   /* workspace missing or smaller than required   */

/* ---- device-side error bits (ORed into *err_word) --------------------- */
#define PKV_DEV_ERR_PAGE 0x1    /* page id outside [0, num_pages)             */
#define PKV_DEV_ERR_SEQ_LEN 0x2 /* active row seq_len outside [1, max_pages*ps] */
#define PKV_DEV_ERR_SLOT 0x4    /* active row slot outside [0, num_slots)     */
#define PKV_DEV_ERR_TIMEOUT 0x8 /* a bounded wait on an async copy gave up    */
#define PKV_DEV_ERR_LOGITS 0x10 /* NaN or +inf logit in an active row         */
#define PKV_DEV_ERR_HISTORY 0x20 /* negative token-history length             */
#define PKV_DEV_ERR_INDPTR 0x40  /* qo_indptr not 0-based, not non-decreasing,
                                    or past the packed token count            */

/* ---- out_kind codes ("Adding a Model", section "How a program runs":
 *      out_kind is audio frame, stop, or other) ------------------------- */
#define PKV_KIND_OTHER 0
#define PKV_KIND_AUDIO 1
#define PKV_KIND_STOP 2

/* Codebook channels of a frame whose stop/continue sample said stop. */
#define PKV_CODE_PAD (-1)

/* Geometry of the paged cache: one bf16 tensor
 *   cache[num_layers][num_pages][2][page_size][num_kv_heads][head_dim]
 * for all layers ("Adding a Model", section "1. The model code").  Index 0
 * of dim 2 holds K, index 1 holds V. */
typedef struct {
  int32_t num_layers;
  int32_t num_pages;
  int32_t page_size;    /* tokens per page: a multiple of 16, at most 1024
                           (16 as in vox-serve, 128 as in mstar's pools)    */
  int32_t num_kv_heads;
  int32_t head_dim;     /* 64 or 128                                         */
} pkv_cache_t;

/* Library version string, e.g. "pkv 0.1.0 sm_103a". */
const char *pkv_version(void);

/* Human-readable name of a status code. */
const char *pkv_error_string(int status);

/* Number of device-side error bits defined above (for binding checks). */
int pkv_num_dev_error_bits(void);

/* The CUDA runtime error code (a cudaError_t value) behind the calling
 * thread's most recent PKV_ERR_CUDA, or the launch error still pending on
 * this thread; 0 when there is none.  A fault in a kernel (an illegal or
 * misaligned address, an illegal instruction) is sticky: every later call
 * in the same CUDA context reports it too.  Host only, no device work. */
int pkv_last_cuda_error(void);

/* The CUDA runtime's name for an error code, e.g. "cudaErrorIllegalAddress"
 * (a static string owned by the CUDA runtime). */
const char *pkv_cuda_error_name(int code);

/* pkv_selftest_wait_timeout -- a diagnostic, not part of the decode step.
 * Every wait of the library's kernels (an mbarrier that a bulk copy or
 * another warp completes) is bounded: when it runs out, the kernel sets
 * PKV_DEV_ERR_TIMEOUT in the error word, stops waiting and returns, and the
 * CUDA context stays usable.  This call runs that same bounded wait in one
 * thread block on an mbarrier that nothing completes, so that the give-up
 * path can be exercised without any fault: after it, *err_word has
 * PKV_DEV_ERR_TIMEOUT set.
 *   limit_ns   the wait's limit, 1 .. 1e9 nanoseconds (else
 *              PKV_ERR_INVALID_ARG).
 *   err_word   device int32, OR-ed into; not NULL. */
int pkv_selftest_wait_timeout(unsigned long long limit_ns, int32_t *err_word,
                              void *stream);

/* ------------------------------------------------------------------------
 * pkv_kv_append -- set_kv_cache(kv_cache, k, v) of "Adding a Model",
 * section "1. The model code": write each row's new key and value into the
 * slot of layer `layer` that holds position seq_lens[b] - 1.
 *
 *   cache       bf16, the layout of pkv_cache_t; written in place.
 *   k, v        bf16 [batch][num_kv_heads][head_dim], the new token's K, V.
 *   page_table  int32 [batch][max_pages]; page_table[b][i] is the page that
 *               holds positions [i*page_size, (i+1)*page_size) of row b.
 *   seq_lens    int32 [batch]; the row's length INCLUDING this token.
 *   active      int32 [batch]; 0 marks a padding entry.
 *
 * An active row writes cache[layer][page][0|1][(n-1) % page_size] with
 * page = page_table[b][(n-1) / page_size], n = seq_lens[b].  A padding row
 * writes its (ignored) k, v to page 0, slot 0, the dummy page, and nowhere
 * else.  Nothing else in the cache changes.
 * Errors: PKV_ERR_INVALID_ARG for a null pointer, batch <= 0, layer outside
 * [0, num_layers), max_pages <= 0 or a bad geometry; PKV_ERR_UNSUPPORTED for
 * num_kv_heads * head_dim not a multiple of 8.  Device: PKV_DEV_ERR_SEQ_LEN
 * or PKV_DEV_ERR_PAGE, and that row writes nothing.
 * ---------------------------------------------------------------------- */
int pkv_kv_append(const pkv_cache_t *geom, void *cache, int layer,
                  const void *k, const void *v, const int32_t *page_table,
                  int max_pages, const int32_t *seq_lens,
                  const int32_t *active, int batch, int32_t *err_word,
                  void *stream);

/* Workspace (bytes) pkv_paged_decode_attn needs for these sizes. */
size_t pkv_decode_workspace_bytes(int batch, int num_qo_heads, int head_dim,
                                  int max_pages, int page_size);

/* ------------------------------------------------------------------------
 * pkv_paged_decode_attn -- attn_wrapper.run(q, kv_cache) of "Adding a
 * Model", section "1. The model code": grouped-query decode attention of one
 * query token per row over that row's pages of layer `layer`.
 *
 * For row b, q head h, kv head g = h / (num_qo_heads / num_kv_heads) (section
 * "2. The program" gives only the head counts; contiguous groups are the
 * reading taken), n = seq_lens[b]:
 *     s_t = sm_scale * <q[b][h], K_t>,   t = 0 .. n-1 (gathered via the
 *                                         page table),
 *     out[b][h] = sum_t softmax(s)_t * V_t,   lse[b][h] = log sum_t e^{s_t}.
 *
 *   q           bf16 [batch][num_qo_heads][head_dim].
 *   sm_scale    softmax scale; pass 1/sqrt(head_dim) for the usual one.
 *   out         [batch][num_qo_heads][head_dim], bf16 (rounded once, to
 *               nearest even) or fp32 when out_fp32 != 0.
 *   lse         fp32 [batch][num_qo_heads] natural-log log-sum-exp, or NULL.
 *   workspace   device scratch of at least pkv_decode_workspace_bytes(...)
 *               bytes (split partials); contents need not be initialised.
 *               Calls that overlap on the device must not share it.
 * Arithmetic: bf16 inputs, fp32 accumulation, long rows split into fixed
 * 512-token pieces merged by log-sum-exp in split order, so the result of a
 * row depends on its own inputs only (not on the batch it is in).
 * Padding rows (active == 0) read nothing and write zeros (lse = -inf).
 * Errors: PKV_ERR_INVALID_ARG (null pointer, bad sizes, num_qo_heads not a
 * multiple of num_kv_heads), PKV_ERR_UNSUPPORTED (head_dim not 64 / 128,
 * page_size not a multiple of 16 or above 1024, more than 64 q heads per kv
 * head), PKV_ERR_WORKSPACE.
 * Device: PKV_DEV_ERR_SEQ_LEN (row written as zeros), PKV_DEV_ERR_PAGE (page 0
 * read instead; row unspecified), PKV_DEV_ERR_TIMEOUT.
 * ---------------------------------------------------------------------- */
int pkv_paged_decode_attn(const pkv_cache_t *geom, const void *cache,
                          int layer, const void *q, int num_qo_heads,
                          float sm_scale, const int32_t *page_table,
                          int max_pages, const int32_t *seq_lens,
                          const int32_t *active, int batch, void *out,
                          int out_fp32, float *lse, void *workspace,
                          size_t workspace_bytes, int32_t *err_word,
                          void *stream);

/* ------------------------------------------------------------------------
 * pkv_paged_decode_attn_static -- pkv_paged_decode_attn for callers that
 * cannot hand the library any device scratch.  (The source pages have no
 * counterpart: this is an addition of this library.)
 *
 * Some hosts can pass device pointers for their own tensors but have no
 * device allocator to offer -- a plugin inside another framework, a foreign
 * language runtime, or a serving engine that reserves all device memory at
 * start-up and allows no allocation afterwards.  This entry point takes the
 * same arguments as pkv_paged_decode_attn minus the workspace and uses a
 * scratch array of PKV_ATTN_STATIC_SCRATCH_BYTES that the library keeps in
 * device memory (a file-scope __device__ array: every GPU that loads the
 * library holds it until the process exits).  It allocates and frees
 * nothing.
 *
 *   - The first call in each CUDA context (normally once per device; again
 *     after cudaDeviceReset makes a new one) looks up the array's device
 *     address (cudaGetSymbolAddress with that device current) and remembers
 *     it; host threads share that lookup safely.  Make the first call on a
 *     device before any stream capture begins.
 *   - Arguments are checked first, exactly as for pkv_paged_decode_attn;
 *     then problems whose pkv_decode_workspace_bytes(...) exceeds
 *     PKV_ATTN_STATIC_SCRATCH_BYTES are rejected with PKV_ERR_WORKSPACE,
 *     before anything is launched.
 *   - All calls share the one array, which keeps the last call's contents
 *     (nothing in it needs to start at zero): calls that can overlap on the
 *     GPU (other streams, other host threads) race on it; serialise them.
 * Results are bit-identical to pkv_paged_decode_attn on the same inputs.
 * ---------------------------------------------------------------------- */
#define PKV_ATTN_STATIC_SCRATCH_BYTES (32u << 20) /* 32 MiB */

int pkv_paged_decode_attn_static(const pkv_cache_t *geom, const void *cache,
                                 int layer, const void *q, int num_qo_heads,
                                 float sm_scale, const int32_t *page_table,
                                 int max_pages, const int32_t *seq_lens,
                                 const int32_t *active, int batch, void *out,
                                 int out_fp32, float *lse, int32_t *err_word,
                                 void *stream);

/* ------------------------------------------------------------------------
 * pkv_decode_plan / pkv_paged_decode_attn_planned -- the same attention as
 * pkv_paged_decode_attn, with its schedule made once for all of a step's
 * layers.  "Supported Models" (sections "Nemotron VoiceChat (nemotron_duplex)
 * notes" and "Chatterbox notes") declare an attention plan on the paged
 * cache, shared by a step's layers and by the captured decode graph of a
 * batch size; the reading taken is that the plan depends on the batch's
 * rows and lengths only, so one plan serves every layer of the step.
 *
 * pkv_decode_plan writes into `workspace` the schedule of a batch: which
 * 512-token splits of which rows form the attention units, longest first.
 * It reads seq_lens and active (on the device, in stream order) and nothing
 * else.  Arguments as for pkv_paged_decode_attn; the cache, q and output
 * are not needed.
 *
 * pkv_paged_decode_attn_planned then runs one layer's attention on that
 * schedule, without the planner: the same arguments as
 * pkv_paged_decode_attn.  The workspace must hold a plan that
 * pkv_decode_plan wrote, earlier in the same stream, with the same geom,
 * num_qo_heads, max_pages, batch and the same contents of seq_lens and
 * active (the caller's contract; the library cannot check it).  Any number
 * of planned calls may follow one plan; each leaves the plan ready for the
 * next.  Results are bit-identical to pkv_paged_decode_attn on the same
 * inputs.  A row that pkv_decode_plan reported as malformed
 * (PKV_DEV_ERR_SEQ_LEN) is reported by the plan only, once per step.  If a
 * row's length changes after the plan so that a planned unit no longer lies
 * inside it (or inside max_pages), the planned call reads nothing for that
 * unit, writes no partial for it and reports PKV_DEV_ERR_SEQ_LEN; that row's
 * output is then undefined, and nothing outside the call's buffers is read
 * or written.
 * Errors: as for pkv_paged_decode_attn.
 * ---------------------------------------------------------------------- */
int pkv_decode_plan(const pkv_cache_t *geom, int num_qo_heads, int max_pages,
                    const int32_t *seq_lens, const int32_t *active, int batch,
                    void *workspace, size_t workspace_bytes, int32_t *err_word,
                    void *stream);

int pkv_paged_decode_attn_planned(const pkv_cache_t *geom, const void *cache,
                                  int layer, const void *q, int num_qo_heads,
                                  float sm_scale, const int32_t *page_table,
                                  int max_pages, const int32_t *seq_lens,
                                  const int32_t *active, int batch, void *out,
                                  int out_fp32, float *lse, void *workspace,
                                  size_t workspace_bytes, int32_t *err_word,
                                  void *stream);

/* ------------------------------------------------------------------------
 * Prefill and mixed steps ("Adding a Model", "How a program runs": lm_prefill
 * runs prompt rows, one graph per row bucket; "Supported Models", Qwen3.5 /
 * Qwen3.8 notes: text prefill and mixed steps, replayed by total tokens).
 * A step's new tokens are packed: request b owns rows
 * [qo_indptr[b], qo_indptr[b+1]) of k, v, q and out (q_b of them), and with
 * n_b = seq_lens[b] (counting them) its token i sits at position
 * n_b - q_b + i.  A decode row is q_b = 1.  qo_indptr int32 [batch + 1],
 * qo_indptr[0] = 0, non-decreasing, qo_indptr[batch] <= total_tokens (rows
 * past it are not touched).  Padding requests (active == 0) write their
 * tokens to page 0, slot 0 and get zero outputs.
 * ---------------------------------------------------------------------- */

/* pkv_kv_append_tokens -- every new token's k, v (bf16 [total_tokens][Hkv]
 * [head_dim]) into the slot of its position in layer `layer`.  Errors as
 * pkv_kv_append; device: PKV_DEV_ERR_SEQ_LEN (request with seq_len < q_b,
 * seq_len < 1 or past max_pages * page_size: it writes nothing),
 * PKV_DEV_ERR_PAGE, PKV_DEV_ERR_INDPTR (a token row that no request owns
 * writes nothing). */
int pkv_kv_append_tokens(const pkv_cache_t *geom, void *cache, int layer,
                         const void *k, const void *v, int total_tokens,
                         const int32_t *qo_indptr, const int32_t *page_table,
                         int max_pages, const int32_t *seq_lens,
                         const int32_t *active, int batch, int32_t *err_word,
                         void *stream);

/* Workspace (bytes) pkv_prefill_attn needs for `batch` requests. */
size_t pkv_prefill_workspace_bytes(int batch);

/* pkv_prefill_attn -- causal grouped-query attention of the new tokens over
 * the paged cache of layer `layer` (after pkv_kv_append_tokens): the token
 * at position p of request b, q head h, attends to positions [0, p] of b
 * with kv head h / (num_qo_heads / num_kv_heads):
 *     out[t][h] = sum_j softmax_j(sm_scale * q[t][h] . K_j) V_j
 *   q    bf16 [total_tokens][num_qo_heads][head_dim] (16-byte aligned)
 *   out  bf16 [total_tokens][num_qo_heads][head_dim] (rounded to nearest
 *        even once, from fp32 accumulation)
 *   lse  fp32 [total_tokens][num_qo_heads] natural-log log-sum-exp, or NULL
 * Tensor cores (tcgen05, bf16 operands, fp32 accumulation in tensor
 * memory); a row's result depends on its own request only.  head_dim 64 or
 * 128, page_size a multiple of 16 up to 1024, up to 128 q heads per kv head.
 * Errors: PKV_ERR_INVALID_ARG (also for sm_scale <= 0 or NaN),
 * PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE.
 * Device: PKV_DEV_ERR_SEQ_LEN (rows written as zeros), PKV_DEV_ERR_PAGE
 * (page 0 read instead), PKV_DEV_ERR_INDPTR, PKV_DEV_ERR_TIMEOUT. */
int pkv_prefill_attn(const pkv_cache_t *geom, const void *cache, int layer,
                     const void *q, int num_qo_heads, float sm_scale,
                     int total_tokens, const int32_t *qo_indptr,
                     const int32_t *page_table, int max_pages,
                     const int32_t *seq_lens, const int32_t *active, int batch,
                     void *out, float *lse, void *workspace,
                     size_t workspace_bytes, int32_t *err_word, void *stream);

/* Workspace (bytes) pkv_seeded_sample needs for these sizes. */
size_t pkv_sample_workspace_bytes(int batch, int vocab);

/* ------------------------------------------------------------------------
 * pkv_seeded_sample -- sample_into of "Adding a Model" (sections "How a
 * program runs" and "2. The program") with the sampler semantics of
 * "Supported Models" (mstar docs), "Fish Audio S2-Pro notes" and
 * "Chatterbox notes".
 *
 * For each active row b with slot s = slots[b]:
 *   - temperature[s] <= 1e-5: greedy, the lowest id among the largest logits;
 *   - else x = logit / temperature[s] (fp64); order tokens by (x desc, id
 *     asc); keep the first top_k[s] (0 or >= vocab: all); then, if
 *     top_p[s] < 1, keep token r of that order iff r == 0 or
 *     S_{r-1} < top_p * Z, where S is the running sum of exp(x - x_max) in
 *     order and Z its total over the top-k survivors (the crossing token is
 *     kept);
 *   - the sample is the kept token with the largest x + g, g = -log(-log u),
 *     u = (2 * (w >> 12) + 1) * 2^-53, w = word 0 of Philox4x64-10 with key
 *     (seeds[s], salt) and counter (token id, steps[s], 0, 0); lowest id on
 *     exact ties.  All of this is computed in fp64.
 *   - out_kind: PKV_KIND_STOP if the token is in stop_tokens, else
 *     PKV_KIND_AUDIO if audio_lo <= token < audio_hi, else PKV_KIND_OTHER.
 *   - advance != 0: steps[s] += 1 after sampling.
 * Padding rows: out_tok = 0, out_kind = OTHER, no state touched.
 *
 *   logits       fp32, row b at logits + b * row_stride (row_stride >= vocab;
 *                4-byte aligned).
 *   slots        int32 [batch]; active int32 [batch].
 *   seeds        uint64 [num_slots]; steps int64 [num_slots] (read, and
 *                written when advance); temperature fp32, top_k int32,
 *                top_p fp32 [num_slots].
 *   stop_tokens  int32 [n_stop] device array, or NULL when n_stop == 0.
 *   out_tok, out_kind  int32 [batch].
 *   workspace    at least pkv_sample_workspace_bytes(batch, vocab) bytes.
 * The result of a row depends on its own logits and slot state only; it is
 * bit-identical whatever batch size or batch position it is sampled at.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_WORKSPACE.  Device: PKV_DEV_ERR_SLOT
 * (row gives token 0, OTHER, no state touched), PKV_DEV_ERR_LOGITS.
 * ---------------------------------------------------------------------- */
int pkv_seeded_sample(const float *logits, int64_t row_stride, int batch,
                      int vocab, const int32_t *slots, const int32_t *active,
                      int num_slots, const uint64_t *seeds, int64_t *steps,
                      const float *temperature, const int32_t *top_k,
                      const float *top_p, uint32_t salt, int advance,
                      const int32_t *stop_tokens, int n_stop,
                      int32_t audio_lo, int32_t audio_hi, int32_t *out_tok,
                      int32_t *out_kind, void *workspace,
                      size_t workspace_bytes, int32_t *err_word,
                      void *stream);

/* ------------------------------------------------------------------------
 * The further sampler settings of a program ("Adding a Model", section
 * "2. The program": min_p, repetition_penalty, repetition_window) and the
 * log-probs it may ask for ("Supported Models", "Qwen3.5 / Qwen3.8":
 * enable_logprobs, and "logprobs_mode": "processed"), applied in the order
 * of that page's Chatterbox notes with top-k before min_p.  Every pointer
 * may be NULL, which turns that control off.  All arrays are device
 * memory.
 *
 *   min_p        fp32 [num_slots]: after top-k, keep rank r >= 1 only while
 *                exp(x_r - x_max) >= min_p[s] (the ranks that pass form a
 *                prefix of the order; <= 0 is off).
 *   rep_penalty  fp32 [num_slots]: before temperature, each distinct token
 *                of the slot's penalty window has its logit divided by the
 *                penalty when positive and multiplied by it otherwise (fp32,
 *                correctly rounded); 1 is off.
 *   rep_window   int32 [num_slots]: the window is the last
 *                min(rep_window[s], hist_len[s], hist_cap) sampled tokens
 *                (a negative window, or NULL: min(hist_len[s], hist_cap)).
 *   history      int32 [num_slots][hist_cap]: the slot's sampled tokens as
 *                a ring, token n of the slot at n % hist_cap; with advance,
 *                the new token is stored at hist_len[s] % hist_cap and
 *                hist_len[s] incremented.  NULL: no penalty, nothing stored.
 *   hist_len     int32 [num_slots] (required with history; a negative
 *                entry raises PKV_DEV_ERR_HISTORY and that slot's row is
 *                sampled without penalty and stores nothing).
 *   hist_cap     ring capacity (> 0 with history).
 *   logprob_raw  fp32 [batch]: log-softmax of the unprocessed logits at the
 *                sampled token.
 *   logprob_proc fp32 [batch]: log of the sampled token's probability in
 *                the distribution it was drawn from (after penalty,
 *                temperature, top-k, min_p and top-p, renormalised over the
 *                kept tokens); 0 for greedy rows.
 * Both log-probs are computed in fp64 and rounded to fp32 (the raw
 * normaliser's terms within 3e-9 of themselves); padding rows get 0.
 * ---------------------------------------------------------------------- */
typedef struct pkv_sample_ext {
  const float *min_p;
  const float *rep_penalty;
  const int32_t *rep_window;
  int32_t *history;
  int32_t *hist_len;
  int32_t hist_cap;
  float *logprob_raw;
  float *logprob_proc;
} pkv_sample_ext_t;

/* Workspace (bytes) pkv_seeded_sample_ext needs for these sizes (enough for
 * any settings; pkv_sample_workspace_bytes suffices when no row can be
 * penalised, i.e. history or rep_penalty is NULL). */
size_t pkv_sample_ext_workspace_bytes(int batch, int vocab);

/* ------------------------------------------------------------------------
 * pkv_seeded_sample_ext -- pkv_seeded_sample with the settings of
 * pkv_sample_ext_t, applied in the order repetition penalty, temperature,
 * top-k, min_p, top-p (top-p renormalised over the tokens that pass top-k
 * and min_p), then the same Gumbel-max draw.  ext == NULL, or all its
 * pointers NULL, is exactly pkv_seeded_sample.  Arguments and results
 * otherwise as for pkv_seeded_sample; the struct itself is read on the host
 * during the call.  Two active rows must not share a slot.
 * Errors: as pkv_seeded_sample; PKV_ERR_INVALID_ARG also for history
 * without hist_len or with hist_cap <= 0, and for misaligned arrays.
 * Device: as pkv_seeded_sample, and PKV_DEV_ERR_HISTORY.
 * ---------------------------------------------------------------------- */
int pkv_seeded_sample_ext(const float *logits, int64_t row_stride, int batch,
                          int vocab, const int32_t *slots,
                          const int32_t *active, int num_slots,
                          const uint64_t *seeds, int64_t *steps,
                          const float *temperature, const int32_t *top_k,
                          const float *top_p, uint32_t salt, int advance,
                          const int32_t *stop_tokens, int n_stop,
                          int32_t audio_lo, int32_t audio_hi,
                          int32_t *out_tok, int32_t *out_kind,
                          const pkv_sample_ext_t *ext, void *workspace,
                          size_t workspace_bytes, int32_t *err_word,
                          void *stream);

/* Workspace (bytes) pkv_codebook_frame_sample needs for these sizes. */
size_t pkv_frame_workspace_bytes(int n_codebooks, int batch, int vocab);

/* ------------------------------------------------------------------------
 * pkv_codebook_frame_sample -- the frame-local codebook loop of
 * MOSS-TTS-Local on SGLang-Omni (mosi.cn blog): per frame, the RVQ
 * codebooks are sampled in order, each one fed back before the next, on a
 * seeded GPU sampler ("AR Engine" section).
 *
 * For each active row b (slot s), for j = 0 .. n_codebooks-1 in order:
 *     logits_j = base[j][b]                           (j == 0 or fb NULL)
 *     logits_j = fl32(base[j][b] + fb[j][code_{j-1}])  (otherwise)
 *     code_j   = the pkv_seeded_sample rule on logits_j with salt 1 + j and
 *                the frame's step steps[s]
 * then steps[s] += 1 (once per frame) and out_kind[b] = PKV_KIND_AUDIO.
 * No trained local transformer exists here: the additive row gather is a
 * synthetic stand-in that keeps the loop serial and data-dependent.
 * Padding rows: codes 0, kind OTHER, no state touched.  One launch per
 * frame; the 12-step loop runs inside the kernel.
 *
 *   base        fp32 [n_codebooks][batch][vocab].
 *   fb          fp32 [n_codebooks][vocab][vocab] or NULL.
 *   out_codes   int32 [batch][n_codebooks]; out_kind int32 [batch].
 *   other arguments as for pkv_seeded_sample.
 * Errors: as pkv_seeded_sample.
 * ---------------------------------------------------------------------- */
int pkv_codebook_frame_sample(const float *base, const float *fb,
                              int n_codebooks, int batch, int vocab,
                              const int32_t *slots, const int32_t *active,
                              int num_slots, const uint64_t *seeds,
                              int64_t *steps, const float *temperature,
                              const int32_t *top_k, const float *top_p,
                              int32_t *out_codes, int32_t *out_kind,
                              void *workspace, size_t workspace_bytes,
                              int32_t *err_word, void *stream);

/* Workspace (bytes) pkv_frame_sample needs for these sizes. */
size_t pkv_frame_sample_workspace_bytes(int n_codebooks, int batch, int vocab,
                                        int ctrl_vocab);

/* ------------------------------------------------------------------------
 * pkv_frame_sample -- a full frame row of MOSS-TTS-Local on SGLang-Omni
 * (mosi.cn blog, section on the model): per frame, the local transformer
 * first gives a stop/continue decision, then the codebooks are sampled in
 * order; a frame row has 1 + n_codebooks channels, channel 0 the control
 * token and the rest the codes (the "[T, 13]" rows); the 13 samplings of a
 * frame run on a seeded GPU sampler ("AR Engine" section).
 *
 * For each active row b (slot s), at the frame's step steps[s]:
 *     out_rows[b][0] = the pkv_seeded_sample rule on ctrl_logits[b] with
 *                      salt 0 and the slot's temperature / top-k / top-p;
 *     if it is stop_ctrl: out_rows[b][1..] = PKV_CODE_PAD, nothing else is
 *                      sampled, out_kind[b] = PKV_KIND_STOP;
 *     else:            out_rows[b][1 + j] = code_j of
 *                      pkv_codebook_frame_sample (salts 1 .. n_codebooks),
 *                      out_kind[b] = PKV_KIND_AUDIO;
 * then steps[s] += 1 (once per frame, stopped or not).  No trained local
 * transformer exists here: the control logits are the caller's, and the
 * control token does not feed the codebooks.  Padding rows: zeros, kind
 * OTHER, no state touched.  One launch per frame.
 *
 *   ctrl_logits fp32 [batch][ctrl_vocab], 4-byte aligned.
 *   stop_ctrl   the control token that means stop, in [0, ctrl_vocab).
 *   out_rows    int32 [batch][1 + n_codebooks].
 *   other arguments as for pkv_codebook_frame_sample.
 * Errors: as pkv_codebook_frame_sample; PKV_ERR_INVALID_ARG also for a
 * NULL ctrl_logits or a stop_ctrl outside [0, ctrl_vocab).
 * ---------------------------------------------------------------------- */
int pkv_frame_sample(const float *ctrl_logits, int ctrl_vocab, int32_t stop_ctrl,
                     const float *base, const float *fb, int n_codebooks,
                     int batch, int vocab, const int32_t *slots,
                     const int32_t *active, int num_slots,
                     const uint64_t *seeds, int64_t *steps,
                     const float *temperature, const int32_t *top_k,
                     const float *top_p, int32_t *out_rows, int32_t *out_kind,
                     void *workspace, size_t workspace_bytes,
                     int32_t *err_word, void *stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* PKV_H_ */
