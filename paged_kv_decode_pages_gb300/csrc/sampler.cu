// sampler.cu -- seeded temperature / top-k / top-p sampling (sample_into of
// "Adding a Model", vox-serve docs) and the frame-local codebook loop
// (MOSS-TTS-Local on SGLang-Omni, mosi.cn blog).
//
// Semantics ("Supported Models", mstar docs, "Fish Audio S2-Pro notes" and
// "Chatterbox notes"): temperature first; top-k then top-p over the tempered
// probabilities of the top-k survivors; the top-p boundary keeps the token
// whose probability carries the running total past top-p; temperature
// <= 1e-5 is greedy; a top-k of 0 or >= vocab is no filter.  Randomness:
// Gumbel-max with Philox4x64-10 (Salmon et al., SC 2011) keyed by
// (seed, salt) at counter (token, step, 0, 0), so a row's sample depends on
// its own logits and slot state only.
//
// Arithmetic.  The definition is stated in fp64 (x = logit / T, e^(x - max),
// prefix sums, x + Gumbel noise).  On this GPU one fp64 warp instruction
// takes as much issue time as several dozen fp32 ones, so the kernels work
// in double-float arithmetic (unevaluated sums of two fp32 values, 48-bit
// significands) and use fp64 only where a decision has to reproduce the
// definition bit for bit:
//  * e^(x - m) = 2^(logit * log2(e) / T - t_max) by Tang's table-driven
//    method (ACM TOMS 15(2), 1989): 2^k * 2^(j/32) * 2^r with |r| <= 1/64, a
//    double-float table of 2^(j/32) and a degree-4 Taylor polynomial for
//    2^r - 1; each term is within 3e-9 of itself.  Normalisers and prefix
//    sums are double-float sums and top-p cuts compare double-float values,
//    so a cut can differ from the fp64 definition only where a prefix sum
//    lies within ~1e-8 of p * Z (a near-tie).
//  * Gumbel-max: scores x + g are first formed in fp32 (absolute error below
//    1.3e-5 + 2.5e-7 |score|).  When another candidate lies within
//    1e-4 + 1e-6 |best| of the best, the contenders are scored again in fp64
//    exactly as the definition states, so the token is the definition's.
//
// Structure:
//  * order key: the fp32 logit mapped to a uint32 that sorts like the float
//    (-0 folded onto +0); composite = key << 32 | ~token, so a larger
//    composite comes first in (value desc, id asc) order, and composites
//    are unique and non-zero.
//  * chunk pass (one CTA per 8192-token chunk of a row): chunk maximum; the
//    chunk's nc largest composites (radix select over 8-bit digits), sorted,
//    nc = min(top-k or 512, max(64, ceil((top-k or 512) / chunks)));
//    for top-p over the whole vocabulary, the partial normaliser
//    z = sum 2^(t - t_max), t = logit * log2(e) / T, as a double-float; for
//    "keep everything", the chunk's Gumbel winner.  The chunking depends on
//    the vocabulary only.
//  * finish (one CTA per row): takes the union of the chunks' candidates and
//    extracts its sorted prefix block by block (radix select of the block's
//    last element, then a sort of the block) only as far as the decision
//    reads: the top-k, or the top-p crossing.  The extracted prefix is the
//    exact global order unless some chunk's last candidate lies strictly
//    inside it while the chunk holds more tokens; then (and for top-k > 512
//    or a crossing past 512 tokens) the row takes an exact general path that
//    streams the row: radix select of the top-k threshold and progressive
//    sorted extraction until the top-p crossing.
//  * the frame kernel runs the same chunk pass and finish for each of the
//    codebooks in turn inside one CTA per row.
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int SB = 256;                 // threads per sampler CTA
constexpr int NW = SB / 32;             // warps per sampler CTA
constexpr int CHUNK = 8192;             // tokens per chunk
constexpr int EPT = CHUNK / SB;         // tokens per thread in a chunk pass
constexpr int NCAND = 64;               // least candidates kept per chunk
constexpr int MAXK_FAST = 512;          // longest prefix the finish extracts
constexpr int CAND_CAP = MAXK_FAST;     // most candidates kept per chunk
constexpr int MAX_CHUNKS = 64;          // vocab <= 64 * 8192
constexpr int UNION_CAP = MAX_CHUNKS * NCAND;  // >= chunks * nc for every vocab
constexpr int GEN_BLOCK = MAXK_FAST;    // sorted block of the general path

enum Mode : int { MODE_GREEDY = 0, MODE_TOPK_SMALL = 1, MODE_TOPP_FULL = 2, MODE_ALL = 3, MODE_GENERAL = 4 };

struct ChunkRec {
  uint64_t top1;       // largest composite of the chunk (0: chunk empty)
  float zh, zl;        // MODE_TOPP_FULL: sum over the chunk of 2^(t - t_top1)
  float ga;            // MODE_ALL: the chunk's best fp32 score
  int32_t gid;         // MODE_ALL: the chunk's winner
  double gscore;       // MODE_ALL: its fp64 score when gexact
  int32_t gexact;      // MODE_ALL: gid was decided among several contenders in fp64
  int32_t ncand;       // candidates kept (sorted, largest first)
  uint64_t cand[CAND_CAP];
  uint64_t pad_[3];
};
static_assert(sizeof(ChunkRec) % 64 == 0, "ChunkRec");

struct RowParams {
  float temperature;
  int32_t top_k;
  float top_p;
  uint32_t salt;
  uint64_t seed;
  int64_t step;
  int K;           // top-k count after normalisation (V when off)
  int mode;
  int nc;          // candidates per chunk
  float c2h, c2l;  // log2(e) / T as a double-float
};

// ---------------------------------------------------------------------------
// double-float arithmetic (Dekker 1971; Knuth TAOCP vol. 2, 4.2.2)
// ---------------------------------------------------------------------------
struct DF {
  float h, l;
};

// s + e == a + b exactly
__device__ __forceinline__ DF df_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}
// the same for |a| >= |b|
__device__ __forceinline__ DF df_fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ DF df_add(DF a, DF b) {
  const DF s = df_two_sum(a.h, b.h);
  return df_fast_two_sum(s.h, __fadd_rn(s.l, __fadd_rn(a.l, b.l)));
}
__device__ __forceinline__ DF df_mul(DF a, DF b) {
  const float p = __fmul_rn(a.h, b.h);
  float e = fmaf(a.h, b.h, -p);
  e = fmaf(a.h, b.l, fmaf(a.l, b.h, e));
  return df_fast_two_sum(p, e);
}
__device__ __forceinline__ DF df_mul_f(DF a, float b) {
  const float p = __fmul_rn(a.h, b);
  return df_fast_two_sum(p, fmaf(a.l, b, fmaf(a.h, b, -p)));
}
__device__ __forceinline__ DF df_div_f(DF a, float b) {
  const float q1 = __fdiv_rn(a.h, b);
  const float r = __fadd_rn(fmaf(-q1, b, a.h), a.l);
  return df_fast_two_sum(q1, __fdiv_rn(r, b));
}
// a < b for normalised double-floats
__device__ __forceinline__ bool df_lt(DF a, DF b) { return a.h < b.h || (a.h == b.h && a.l < b.l); }
__device__ __forceinline__ DF df_shfl_xor(DF v, int m) {
  return {__shfl_xor_sync(FULL_MASK, v.h, m), __shfl_xor_sync(FULL_MASK, v.l, m)};
}
__device__ __forceinline__ DF df_shfl_up(DF v, int d) {
  return {__shfl_up_sync(FULL_MASK, v.h, d), __shfl_up_sync(FULL_MASK, v.l, d)};
}
__device__ __forceinline__ DF df_shfl(DF v, int src) {
  return {__shfl_sync(FULL_MASK, v.h, src), __shfl_sync(FULL_MASK, v.l, src)};
}

// log2(e) and ln(2) as double-floats
constexpr float LOG2E_H = 0x1.715476p+0f, LOG2E_L = 0x1.4ae0c0p-26f;
constexpr float LN2_H = 0x1.62e430p-1f, LN2_L = -0x1.05c610p-29f;

// 2^(j/32), j = 0..31, split into an fp32 value and an fp32 correction
// (each pair is within 4e-15 of 2^(j/32))
__constant__ float c_exp2_tab_h[32] = {
    0x1.000000p+0f, 0x1.059b0ep+0f, 0x1.0b5586p+0f, 0x1.11301ep+0f, 0x1.172b84p+0f,
    0x1.1d4874p+0f, 0x1.2387a6p+0f, 0x1.29e9e0p+0f, 0x1.306fe0p+0f, 0x1.371a74p+0f,
    0x1.3dea64p+0f, 0x1.44e086p+0f, 0x1.4bfdaep+0f, 0x1.5342b6p+0f, 0x1.5ab07ep+0f,
    0x1.6247ecp+0f, 0x1.6a09e6p+0f, 0x1.71f75ep+0f, 0x1.7a1148p+0f, 0x1.82589ap+0f,
    0x1.8ace54p+0f, 0x1.93737cp+0f, 0x1.9c4918p+0f, 0x1.a5503cp+0f, 0x1.ae89fap+0f,
    0x1.b7f770p+0f, 0x1.c199bep+0f, 0x1.cb720ep+0f, 0x1.d5818ep+0f, 0x1.dfc974p+0f,
    0x1.ea4afap+0f, 0x1.f50766p+0f};
__constant__ float c_exp2_tab_l[32] = {
    0.0f,             -0x1.9d4f52p-25f, 0x1.9f3122p-25f,  -0x1.fdb496p-25f, -0x1.c15742p-27f,
    -0x1.d2e8cap-25f, 0x1.ceac48p-25f,  -0x1.5c0424p-25f, 0x1.4636e2p-25f,  -0x1.18aac6p-25f,
    0x1.824684p-25f,  0x1.8624b4p-30f,  -0x1.593abcp-25f, -0x1.2c5610p-25f, -0x1.5bd5ecp-27f,
    -0x1.f8b550p-25f, 0x1.9fcef4p-26f,  0x1.1d8beep-25f,  -0x1.829fd0p-25f, -0x1.accc7cp-26f,
    0x1.15506ep-27f,  -0x1.e64744p-25f, 0x1.51f848p-27f,  -0x1.b83b54p-25f, -0x1.a94b14p-26f,
    -0x1.a09438p-25f, -0x1.3d56b2p-27f, -0x1.8837ccp-27f, -0x1.822dbcp-27f, -0x1.908c94p-25f,
    0x1.52486cp-27f,  -0x1.246eb0p-26f};

// t = v * c2 - tm <= ~0 with c2, tm double-floats
struct Exp2Ctx {
  float c2h, c2l, th, tl;
};

__device__ __forceinline__ Exp2Ctx exp2_ctx(const RowParams &P, float vmax) {
  const DF tm = df_mul_f(DF{P.c2h, P.c2l}, vmax);
  return {P.c2h, P.c2l, tm.h, tm.l};
}

// 2^(v * c2 - tm) as a normalised double-float; 0 below 2^-125 and for a
// -inf v (whose products give NaN and fail the range test).
__device__ __forceinline__ DF df_exp2_rel(float v, const Exp2Ctx &c, const float *tab_h,
                                          const float *tab_l) {
  // v * c2 = ph + pl
  const float ph = __fmul_rn(v, c.c2h);
  const float pl = fmaf(v, c.c2l, fmaf(v, c.c2h, -ph));
  // t = s.h + tlow
  const DF s = df_two_sum(ph, -c.th);
  const float tlow = __fsub_rn(__fadd_rn(s.l, pl), c.tl);
  if (!(s.h > -125.0f)) return {0.0f, 0.0f};
  // n = rint(32 s.h) = 32 k + j; s.h - n / 32 is exact
  const float y = fmaf(s.h, 32.0f, 12582912.0f);
  const int n = __float_as_int(y) - 0x4B400000;
  const float g = fmaf(__fsub_rn(y, 12582912.0f), -0.03125f, s.h);
  const float r = __fadd_rn(g, tlow);
  // 2^r - 1 = u + u^2/2 + u^3/6 + u^4/24, u = r ln 2, |u| < 0.011
  const float u = fmaf(r, LN2_H, __fmul_rn(r, LN2_L));
  float q = fmaf(u, 1.0f / 24.0f, 1.0f / 6.0f);
  q = fmaf(q, u, 0.5f);
  q = fmaf(q, u, 1.0f);
  q = __fmul_rn(q, u);
  const int j = n & 31, k = n >> 5;
  const float t0 = tab_h[j];
  const DF e = df_fast_two_sum(t0, fmaf(t0, q, tab_l[j]));
  const float sc = __int_as_float((k + 127) << 23);  // 2^k, k in [-125, 0]
  return {__fmul_rn(e.h, sc), __fmul_rn(e.l, sc)};
}

// acc += e, keeping the exact rounding error of the high parts
__device__ __forceinline__ void df_accumulate(DF &acc, DF e) {
  const DF s = df_two_sum(acc.h, e.h);
  acc.h = s.h;
  acc.l = __fadd_rn(acc.l, __fadd_rn(s.l, e.l));
}

// ---------------------------------------------------------------------------
// Philox4x64-10 and Gumbel noise
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t philox_word0(uint64_t seed, uint32_t salt, uint64_t token,
                                                 uint64_t step) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
  uint64_t c0 = token, c1 = step, c2 = 0, c3 = 0;
  uint64_t k0 = seed, k1 = salt;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
    const uint64_t hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
    const uint64_t n0 = hi1 ^ c1 ^ k0;
    const uint64_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += W0;
    k1 += W1;
  }
  return c0;
}

// the 52-bit draw m of u = (2m + 1) 2^-53
__device__ __forceinline__ uint64_t gumbel_bits(const RowParams &P, int token) {
  return philox_word0(P.seed, P.salt, (uint64_t)(uint32_t)token, (uint64_t)P.step) >> 12;
}

// g = -log(-log u) as the definition states (fp64)
__device__ __forceinline__ double gumbel_exact(uint64_t m) {
  const double u = (double)(2ull * m + 1ull) * 0x1p-53;
  return -log(-log(u));
}

// the same in fp32: -log u from u itself below 1/2 and from 1 - u (exact in
// integers) above, so that -log u keeps ~2e-7 relative accuracy
__device__ __forceinline__ float gumbel_approx(uint64_t m) {
  float L;
  if (m < (1ull << 51))
    L = -logf(__fmul_rn(__ull2float_rn(2ull * m + 1ull), 0x1p-53f));
  else
    L = -log1pf(-__fmul_rn(__ull2float_rn((1ull << 53) - 2ull * m - 1ull), 0x1p-53f));
  return -logf(L);
}

__device__ __forceinline__ float score_margin(float best) { return 1e-4f + 1e-6f * fabsf(best); }

// ---------------------------------------------------------------------------
// order keys
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float f, bool &bad) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) {  // NaN: report, rank like -inf
    bad = true;
    u = 0xff800000u;
  } else if (u == 0x7f800000u) {
    bad = true;
  }
  if (u == 0x80000000u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  const uint32_t u = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
  return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t composite(uint32_t key, int token) {
  return ((uint64_t)key << 32) | (uint32_t)(~(uint32_t)token);
}
__device__ __forceinline__ int comp_token(uint64_t c) { return (int)(~(uint32_t)c); }
__device__ __forceinline__ float comp_value(uint64_t c) { return key_value((uint32_t)(c >> 32)); }

__device__ __forceinline__ float approx_score(const RowParams &P, uint64_t cc) {
  return __fadd_rn(__fdiv_rn(comp_value(cc), P.temperature),
                   gumbel_approx(gumbel_bits(P, comp_token(cc))));
}
__device__ __forceinline__ double exact_score(const RowParams &P, uint64_t cc) {
  return (double)comp_value(cc) / (double)P.temperature +
         gumbel_exact(gumbel_bits(P, comp_token(cc)));
}

// ---------------------------------------------------------------------------
// shared scratch
// ---------------------------------------------------------------------------
struct SampSmem {
  uint32_t hist[256];
  uint64_t red_u64[NW];
  double red_d[SB];
  int32_t red_i[SB];
  float wf[NW], wh[NW], wl[NW];
  int32_t wi[NW];
  uint64_t sel_prefix;
  uint32_t sel_want;
  uint32_t sel_done;
  uint32_t cnt;
  int32_t flag;
  int32_t token;
  int32_t kept;
  int32_t done;
  float e2h[32], e2l[32];                // the 2^(j/32) table
  uint64_t uni[UNION_CAP];               // finish: the chunks' candidates; chunk pass: its own
  uint64_t pre[MAXK_FAST];               // finish / general path: extracted sorted block(s)
  float esh[MAXK_FAST], esl[MAXK_FAST];  // e^(x - m) of pre as double-floats; fp32 scores
};

__device__ __forceinline__ void load_exp2_table(SampSmem &sm) {
  if (threadIdx.x < 32) {
    sm.e2h[threadIdx.x] = c_exp2_tab_h[threadIdx.x];
    sm.e2l[threadIdx.x] = c_exp2_tab_l[threadIdx.x];
  }
}

// ---------------------------------------------------------------------------
// block primitives (all SB threads must call)
// ---------------------------------------------------------------------------
__device__ uint64_t block_max_u64(uint64_t v, SampSmem &sm) {
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const uint64_t o = __shfl_xor_sync(FULL_MASK, v, off);
    v = o > v ? o : v;
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.red_u64[threadIdx.x >> 5] = v;
  __syncthreads();
  uint64_t r = sm.red_u64[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) r = sm.red_u64[w] > r ? sm.red_u64[w] : r;
  __syncthreads();
  return r;
}

// Double-float sum in a fixed order (xor tree in each warp, then the warps
// in order); every thread gets the result.
__device__ DF block_sum_df(DF v, SampSmem &sm) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v = df_add(v, df_shfl_xor(v, off));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    sm.wh[threadIdx.x >> 5] = v.h;
    sm.wl[threadIdx.x >> 5] = v.l;
  }
  __syncthreads();
  DF r = {sm.wh[0], sm.wl[0]};
#pragma unroll
  for (int w = 1; w < NW; ++w) r = df_add(r, DF{sm.wh[w], sm.wl[w]});
  __syncthreads();
  return r;
}

__device__ int block_sum_i(int v, SampSmem &sm) {
  v = __reduce_add_sync(FULL_MASK, v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.wi[threadIdx.x >> 5] = v;
  __syncthreads();
  int r = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) r += sm.wi[w];
  __syncthreads();
  return r;
}

// Exclusive prefix of per-thread counts in thread order; *total gets the sum.
__device__ int block_excl_scan(int c, SampSmem &sm, int *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(FULL_MASK, incl, off);
    if (lane >= off) incl += o;
  }
  __syncthreads();
  if (lane == 31) sm.wi[w] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    before += (i < w) ? sm.wi[i] : 0;
    all += sm.wi[i];
  }
  __syncthreads();
  *total = all;
  return before + incl - c;
}

// Argmax of (score desc, id asc); ids < 0 mark "none".
__device__ __forceinline__ bool better(double s, int id, double bs, int bid) {
  if (bid < 0) return id >= 0;
  if (id < 0) return false;
  return s > bs || (s == bs && id < bid);
}
__device__ __forceinline__ bool better_f(float s, int id, float bs, int bid) {
  if (bid < 0) return id >= 0;
  if (id < 0) return false;
  return s > bs || (s == bs && id < bid);
}

__device__ int block_argmax(double s, int id, SampSmem &sm, double *best_score = nullptr) {
  __syncthreads();
  sm.red_d[threadIdx.x] = s;
  sm.red_i[threadIdx.x] = id;
  __syncthreads();
  for (int st = SB / 2; st > 0; st >>= 1) {
    if ((int)threadIdx.x < st) {
      const double s2 = sm.red_d[threadIdx.x + st];
      const int i2 = sm.red_i[threadIdx.x + st];
      if (better(s2, i2, sm.red_d[threadIdx.x], sm.red_i[threadIdx.x])) {
        sm.red_d[threadIdx.x] = s2;
        sm.red_i[threadIdx.x] = i2;
      }
    }
    __syncthreads();
  }
  const int r = sm.red_i[0];
  if (best_score) *best_score = sm.red_d[0];
  __syncthreads();
  return r;
}

__device__ int block_argmax_f(float s, int id, SampSmem &sm, float *best_score) {
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float os = __shfl_xor_sync(FULL_MASK, s, off);
    const int oi = __shfl_xor_sync(FULL_MASK, id, off);
    if (better_f(os, oi, s, id)) {
      s = os;
      id = oi;
    }
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    sm.wf[threadIdx.x >> 5] = s;
    sm.wi[threadIdx.x >> 5] = id;
  }
  __syncthreads();
  float bs = sm.wf[0];
  int bid = sm.wi[0];
#pragma unroll
  for (int w = 1; w < NW; ++w)
    if (better_f(sm.wf[w], sm.wi[w], bs, bid)) {
      bs = sm.wf[w];
      bid = sm.wi[w];
    }
  __syncthreads();
  *best_score = bs;
  return bid;
}

// ---------------------------------------------------------------------------
// sorting (descending) of u64 values in shared memory
// ---------------------------------------------------------------------------
// Bitonic network over 32 * E values held E per lane by one warp.
template <int E>
__device__ void warp_sort_desc(uint64_t *v) {
  const int lane = threadIdx.x & 31;
  uint64_t x[E];
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = v[lane * E + e];
#pragma unroll
  for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j < E) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int p = e ^ j;
          if (p > e) {
            const bool desc = ((lane * E + e) & k) == 0;
            const uint64_t a = x[e], b = x[p];
            const bool sw = desc ? (a < b) : (a > b);
            x[e] = sw ? b : a;
            x[p] = sw ? a : b;
          }
        }
      } else {
        const int lj = j / E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const uint64_t o = __shfl_xor_sync(FULL_MASK, x[e], lj);
          const bool lower = (lane & lj) == 0;
          const bool desc = ((lane * E + e) & k) == 0;
          const bool take_max = lower == desc;
          x[e] = take_max ? (o > x[e] ? o : x[e]) : (o < x[e] ? o : x[e]);
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) v[lane * E + e] = x[e];
}

// Bitonic network over n (power of two) values, one compare-exchange pair per
// thread and step.
__device__ void block_sort_desc(uint64_t *v, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int p = threadIdx.x; p < n / 2; p += SB) {
        const int i = ((p & ~(j - 1)) << 1) | (p & (j - 1));  // bit j of i is clear
        const uint64_t a = v[i], b = v[i + j];
        const bool desc = (i & k) == 0;
        if (desc ? (a < b) : (a > b)) {
          v[i] = b;
          v[i + j] = a;
        }
      }
      __syncthreads();
    }
  }
}

// the padded length sort_desc sorts: a power of two, at least 32
__device__ __forceinline__ int sort_width(int n) {
  int n2 = 32;
  while (n2 < n) n2 <<= 1;
  return n2;
}

// Sorts v[0, sort_width(n)) descending; the caller has zero-filled past n.
__device__ void sort_desc(uint64_t *v, int n) {
  const int n2 = sort_width(n);
  __syncthreads();
  if (n2 <= 128) {
    if (threadIdx.x < 32) {
      if (n2 == 32)
        warp_sort_desc<1>(v);
      else if (n2 == 64)
        warp_sort_desc<2>(v);
      else
        warp_sort_desc<4>(v);
    }
    __syncthreads();
  } else {
    block_sort_desc(v, n2);
  }
}

// ---------------------------------------------------------------------------
// radix selection over composites (8-bit digits, most significant first)
// ---------------------------------------------------------------------------
// Warp 0 walks the 256-bin histogram from the top bin down and picks the
// bin holding the `want`-th (1-based) largest element.  Results in sm.
__device__ void select_bin(SampSmem &sm, int shift) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    // lane covers bins 255-8*lane .. 248-8*lane (descending)
    uint32_t c[8];
    uint32_t tot = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      c[e] = sm.hist[255 - 8 * lane - e];
      tot += c[e];
    }
    uint32_t incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL_MASK, incl, off);
      if (lane >= off) incl += o;
    }
    const uint32_t excl = incl - tot;
    const uint32_t want = sm.sel_want;
    const bool mine = excl < want && want <= incl;
    if (mine) {
      uint32_t above = excl;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (above + c[e] >= want) {
          const uint32_t bin = 255 - 8 * lane - e;
          const uint32_t w2 = want - above;
          sm.sel_prefix |= (uint64_t)bin << shift;
          sm.sel_done = (w2 == c[e]) ? 1u : 0u;
          sm.sel_want = w2;
          break;
        }
        above += c[e];
      }
    }
  }
  __syncthreads();
}

// Composite of rank `rank` (0-based, descending) among the non-zero values
// get(i), i < n, that are below `upper`.  Requires that many such values.
template <class Get>
__device__ uint64_t select_rank_of(int n, Get get, uint64_t upper, int rank, SampSmem &sm) {
  __syncthreads();
  if (threadIdx.x == 0) {
    sm.sel_prefix = 0;
    sm.sel_want = (uint32_t)rank + 1u;
    sm.sel_done = 0;
  }
  __syncthreads();
  uint64_t mask = 0;
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += SB) sm.hist[i] = 0;
    __syncthreads();
    const uint64_t prefix = sm.sel_prefix;
    for (int i = threadIdx.x; i < n; i += SB) {
      const uint64_t cc = get(i);
      if (cc != 0ull && cc < upper && (cc & mask) == prefix)
        atomicAdd(&sm.hist[(cc >> shift) & 255u], 1u);
    }
    __syncthreads();
    select_bin(sm, shift);
    mask |= 255ull << shift;
    if (sm.sel_done) break;
  }
  const uint64_t r = sm.sel_prefix;
  __syncthreads();
  return r;
}

// Copies the non-zero values get(i) in [lo, upper) to dst (in no particular
// order; at most cap of them); returns how many there were.
template <class Get>
__device__ int collect_range(int n, Get get, uint64_t lo, uint64_t upper, uint64_t *dst, int cap,
                             SampSmem &sm) {
  int c = 0;
  for (int i = threadIdx.x; i < n; i += SB) {
    const uint64_t cc = get(i);
    c += (cc != 0ull && cc >= lo && cc < upper) ? 1 : 0;
  }
  int total;
  int pos = block_excl_scan(c, sm, &total);
  for (int i = threadIdx.x; i < n && c > 0; i += SB) {
    const uint64_t cc = get(i);
    if (cc != 0ull && cc >= lo && cc < upper) {
      if (pos < cap) dst[pos] = cc;
      ++pos;
      --c;
    }
  }
  __syncthreads();
  return total;
}

// ---------------------------------------------------------------------------
// Gumbel-max over n candidates given by composite (0: none); fp32 scores
// first, the definition's fp64 scores for the contenders when the fp32
// scores cannot separate them.  `store` (nullable) keeps the fp32 scores
// between the passes.
// ---------------------------------------------------------------------------
template <class Get>
__device__ int gumbel_pick(const RowParams &P, int n, Get get, float *store, SampSmem &sm) {
  float bs = 0.0f;
  int bid = -1;
  for (int r = threadIdx.x; r < n; r += SB) {
    const uint64_t cc = get(r);
    if (cc == 0ull) continue;
    const float s = approx_score(P, cc);
    if (store) store[r] = s;
    if (better_f(s, comp_token(cc), bs, bid)) {
      bs = s;
      bid = comp_token(cc);
    }
  }
  float best;
  const int winner = block_argmax_f(bs, bid, sm, &best);
  const float floor_s = best - score_margin(best);
  int c = 0;
  for (int r = threadIdx.x; r < n; r += SB) {
    const uint64_t cc = get(r);
    if (cc != 0ull && (store ? store[r] : approx_score(P, cc)) >= floor_s) ++c;
  }
  if (block_sum_i(c, sm) <= 1) return winner;
  double es = 0.0;
  int eid = -1;
  for (int r = threadIdx.x; r < n; r += SB) {
    const uint64_t cc = get(r);
    if (cc != 0ull && (store ? store[r] : approx_score(P, cc)) >= floor_s) {
      const double x = exact_score(P, cc);
      if (better(x, comp_token(cc), es, eid)) {
        es = x;
        eid = comp_token(cc);
      }
    }
  }
  return block_argmax(es, eid, sm);
}

// ---------------------------------------------------------------------------
// top-p scan (one warp): rank r is kept iff r == 0 or the sum of the kept
// probabilities before it is below p * Z.  Scans es[0, n) of ranks r0 + i
// with the running sum `carry`; returns true when the cut falls inside, with
// *kept = the number kept from this block.
// ---------------------------------------------------------------------------
__device__ bool topp_scan_warp(const float *esh, const float *esl, int n, int r0, DF &carry,
                               DF pz, int *kept) {
  const int lane = threadIdx.x & 31;
  for (int base = 0; base < n; base += 32) {
    const int r = base + lane;
    const DF e = r < n ? DF{esh[r], esl[r]} : DF{0.0f, 0.0f};
    DF inc = e;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const DF o = df_shfl_up(inc, off);
      if (lane >= off) inc = df_add(o, inc);
    }
    DF ex = df_shfl_up(inc, 1);
    if (lane == 0) ex = DF{0.0f, 0.0f};
    const DF S = df_add(carry, ex);
    const bool stop = r < n && r0 + r > 0 && !df_lt(S, pz);
    const unsigned bm = __ballot_sync(FULL_MASK, stop);
    if (bm) {
      *kept = base + __ffs(bm) - 1;
      return true;
    }
    carry = df_add(carry, df_shfl(inc, 31));
  }
  *kept = n;
  return false;
}

// ---------------------------------------------------------------------------
// chunk pass
// ---------------------------------------------------------------------------
__device__ void chunk_pass(const float *__restrict__ row, int V, int c, const RowParams &P,
                           ChunkRec *rec, SampSmem &sm, int32_t *err) {
  const int tid = threadIdx.x;
  const int start = c * CHUNK;
  const int cnt = min(CHUNK, V - start);
  uint32_t key[EPT];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int i = tid + j * SB;
    key[j] = (i < cnt) ? order_key(row[start + i], bad) : 0u;  // may be written by this kernel: no __ldg
  }
  if (bad) report(err, PKV_DEV_ERR_LOGITS);
  uint64_t mine = 0;
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int i = tid + j * SB;
    if (i < cnt) {
      const uint64_t cc = composite(key[j], start + i);
      mine = cc > mine ? cc : mine;
    }
  }
  const uint64_t top1 = block_max_u64(mine, sm);
  if (tid == 0) rec->top1 = top1;
  if (P.mode == MODE_GREEDY || P.mode == MODE_GENERAL) return;

  if (P.mode == MODE_ALL) {
    // the chunk's Gumbel winner: fp32 scores, fp64 among close contenders
    float sa[EPT];
    float bs = 0.0f;
    int bid = -1;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int i = tid + j * SB;
      sa[j] = 0.0f;
      if (i < cnt) {
        sa[j] = approx_score(P, composite(key[j], start + i));
        if (better_f(sa[j], start + i, bs, bid)) {
          bs = sa[j];
          bid = start + i;
        }
      }
    }
    float best;
    const int id = block_argmax_f(bs, bid, sm, &best);
    const float floor_s = best - score_margin(best);
    int n_in = 0;
#pragma unroll
    for (int j = 0; j < EPT; ++j) n_in += (tid + j * SB < cnt && sa[j] >= floor_s) ? 1 : 0;
    if (block_sum_i(n_in, sm) <= 1) {
      if (tid == 0) {
        rec->ga = best;
        rec->gid = id;
        rec->gexact = 0;
      }
      return;
    }
    double es = 0.0;
    int eid = -1;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int i = tid + j * SB;
      if (i < cnt && sa[j] >= floor_s) {
        const double x = exact_score(P, composite(key[j], start + i));
        if (better(x, start + i, es, eid)) {
          es = x;
          eid = start + i;
        }
      }
    }
    double ebest;
    const int ewin = block_argmax(es, eid, sm, &ebest);
    if (tid == 0) {
      rec->ga = best;
      rec->gid = ewin;
      rec->gscore = ebest;
      rec->gexact = 1;
    }
    return;
  }

  // the chunk's nc largest composites
  const int nc = P.nc;
  uint64_t thr = 0;  // keep composites >= thr
  if (cnt > nc) {
    if (tid == 0) {
      sm.sel_prefix = 0;
      sm.sel_want = (uint32_t)nc;
      sm.sel_done = 0;
    }
    __syncthreads();
    uint64_t mask = 0;
    for (int pass = 0; pass < 8; ++pass) {
      const int shift = 56 - 8 * pass;
      for (int i = tid; i < 256; i += SB) sm.hist[i] = 0;
      __syncthreads();
      const uint64_t prefix = sm.sel_prefix;
#pragma unroll
      for (int j = 0; j < EPT; ++j) {
        const int i = tid + j * SB;
        if (i < cnt) {
          const uint64_t cc = composite(key[j], start + i);
          if ((cc & mask) == prefix) atomicAdd(&sm.hist[(cc >> shift) & 255u], 1u);
        }
      }
      __syncthreads();
      select_bin(sm, shift);
      mask |= 255ull << shift;
      if (sm.sel_done) break;
    }
    thr = sm.sel_prefix;
    __syncthreads();
  }
  int mine_c = 0;
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int i = tid + j * SB;
    mine_c += (i < cnt && composite(key[j], start + i) >= thr) ? 1 : 0;
  }
  int got;
  int pos = block_excl_scan(mine_c, sm, &got);
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int i = tid + j * SB;
    if (i < cnt) {
      const uint64_t cc = composite(key[j], start + i);
      if (cc >= thr) {
        if (pos < nc) sm.uni[pos] = cc;
        ++pos;
      }
    }
  }
  got = min(got, nc);
  for (int i = got + tid; i < sort_width(nc); i += SB) sm.uni[i] = 0ull;
  sort_desc(sm.uni, nc);
  for (int i = tid; i < nc; i += SB) rec->cand[i] = sm.uni[i];
  if (tid == 0) rec->ncand = got;

  if (P.mode == MODE_TOPP_FULL) {
    // z = sum over the chunk of 2^(t - t_top1), t = logit * log2(e) / T
    const Exp2Ctx ctx = exp2_ctx(P, comp_value(top1));
    DF acc = {0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < EPT; ++j)
      if (tid + j * SB < cnt) df_accumulate(acc, df_exp2_rel(key_value(key[j]), ctx, sm.e2h, sm.e2l));
    const DF z = block_sum_df(df_fast_two_sum(acc.h, acc.l), sm);
    if (tid == 0) {
      rec->zh = z.h;
      rec->zl = z.l;
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// general path: exact, streams the row (used when the candidates do not decide)
// ---------------------------------------------------------------------------
__device__ int general_sample(const float *__restrict__ row, int V, const RowParams &P,
                              uint64_t top1, SampSmem &sm) {
  const int tid = threadIdx.x;
  const int K = P.K;
  auto rowc = [&](int i) {
    bool dummy = false;
    return composite(order_key(row[i], dummy), i);
  };
  const uint64_t thrK = (K < V) ? select_rank_of(V, rowc, ~0ull, K - 1, sm) : 0ull;
  uint64_t thr = thrK;
  if (P.top_p < 1.0f) {
    const Exp2Ctx ctx = exp2_ctx(P, comp_value(top1));
    DF acc = {0.0f, 0.0f};
    for (int i = tid; i < V; i += SB) {
      const uint64_t cc = rowc(i);
      if (cc >= thrK) df_accumulate(acc, df_exp2_rel(comp_value(cc), ctx, sm.e2h, sm.e2l));
    }
    const DF pz = df_mul_f(block_sum_df(df_fast_two_sum(acc.h, acc.l), sm), P.top_p);
    // progressive sorted extraction until the running sum reaches p * Z
    uint64_t upper = ~0ull;
    int taken = 0;
    DF carry = {0.0f, 0.0f};
    for (;;) {
      const int M = min(GEN_BLOCK, K - taken);
      const uint64_t lo = select_rank_of(V, rowc, upper, M - 1, sm);
      collect_range(V, rowc, lo, upper, sm.pre, GEN_BLOCK, sm);
      for (int i = M + tid; i < sort_width(M); i += SB) sm.pre[i] = 0ull;
      sort_desc(sm.pre, M);
      for (int r = tid; r < M; r += SB) {
        const DF e = df_exp2_rel(comp_value(sm.pre[r]), ctx, sm.e2h, sm.e2l);
        sm.esh[r] = e.h;
        sm.esl[r] = e.l;
      }
      __syncthreads();
      if (tid < 32) {
        int k;
        const bool cut = topp_scan_warp(sm.esh, sm.esl, M, taken, carry, pz, &k);
        if (tid == 0) {
          sm.done = (cut || taken + M >= K) ? 1 : 0;
          // the smallest kept composite: the block's k-th, or for k == 0 the
          // previous block's last (which is `upper`)
          sm.sel_prefix = k > 0 ? sm.pre[k - 1] : upper;
        }
      }
      __syncthreads();
      const bool done = sm.done != 0;
      const uint64_t cutoff = sm.sel_prefix;
      taken += M;
      upper = lo;
      __syncthreads();
      if (done) {
        thr = cutoff;
        break;
      }
    }
  }
  // Gumbel-max over the kept tokens (composite >= thr)
  auto kept_c = [&](int i) {
    const uint64_t cc = rowc(i);
    return cc >= thr ? cc : 0ull;
  };
  return gumbel_pick(P, V, kept_c, nullptr, sm);
}

// ---------------------------------------------------------------------------
// finish: one CTA per row
// ---------------------------------------------------------------------------
__device__ int finish_row(const float *__restrict__ row, int V, int nch, const RowParams &P,
                          const ChunkRec *recs, SampSmem &sm) {
  const int tid = threadIdx.x;
  if (P.mode == MODE_GREEDY) {
    uint64_t best = 0;
    for (int c = 0; c < nch; ++c) best = recs[c].top1 > best ? recs[c].top1 : best;
    return comp_token(best);
  }
  if (P.mode == MODE_ALL) {
    // the chunks' winners; fp64 among those the fp32 scores cannot separate
    float A = 0.0f;
    int aid = -1;
    for (int c = 0; c < nch; ++c)
      if (better_f(recs[c].ga, recs[c].gid, A, aid)) {
        A = recs[c].ga;
        aid = recs[c].gid;
      }
    const float floor_s = A - score_margin(A);
    int n_in = 0;
    for (int c = 0; c < nch; ++c) n_in += recs[c].ga >= floor_s ? 1 : 0;
    if (n_in <= 1) return aid;
    double es = 0.0;
    int eid = -1;
    if (tid < nch && recs[tid].ga >= floor_s) {
      const int tok = recs[tid].gid;
      bool dummy = false;
      es = recs[tid].gexact ? recs[tid].gscore
                            : exact_score(P, composite(order_key(row[tok], dummy), tok));
      eid = tok;
    }
    return block_argmax(es, eid, sm);
  }
  uint64_t top1 = 0;
  for (int c = 0; c < nch; ++c) top1 = recs[c].top1 > top1 ? recs[c].top1 : top1;
  if (P.mode == MODE_GENERAL) return general_sample(row, V, P, top1, sm);

  // the union of the chunks' candidates
  const int nc = P.nc;
  const int nu = nch * nc;
  for (int i = tid; i < nu; i += SB) {
    const int c = i / nc;
    sm.uni[i] = recs[c].cand[i - c * nc];
  }
  if (tid == 0) sm.cnt = 0;
  __syncthreads();
  if (tid < nch) atomicAdd(&sm.cnt, (uint32_t)recs[tid].ncand);
  __syncthreads();
  const int nreal = (int)sm.cnt;
  const bool full = P.mode == MODE_TOPP_FULL;
  const bool topp = P.top_p < 1.0f;
  const int nv = min(full ? MAXK_FAST : P.K, nreal);
  const Exp2Ctx ctx = exp2_ctx(P, comp_value(top1));
  DF pz = {0.0f, 0.0f};
  if (full) {
    // Z: the chunks' partial sums rescaled from their maxima to the row's
    DF zc = {0.0f, 0.0f};
    if (tid < nch && recs[tid].top1 != 0ull)
      zc = df_mul(DF{recs[tid].zh, recs[tid].zl},
                  df_exp2_rel(comp_value(recs[tid].top1), ctx, sm.e2h, sm.e2l));
    pz = df_mul_f(block_sum_df(zc, sm), P.top_p);
  }
  // extract the sorted prefix block by block (64, 128, 256, ... tokens)
  auto uget = [&](int i) { return sm.uni[i]; };
  uint64_t upper = ~0ull;
  DF carry = {0.0f, 0.0f};
  int lo = 0, blk = full ? 64 : nv;
  bool fallback = !full && P.K > nreal;  // some chunk holds top-k tokens it did not give
  int kept = 0;
  while (!fallback) {
    const int hi = min(lo + blk, nv);
    const int M = hi - lo;
    const uint64_t cut = select_rank_of(nu, uget, upper, M - 1, sm);
    collect_range(nu, uget, cut, upper, sm.pre + lo, M, sm);
    for (int i = M + tid; i < sort_width(M); i += SB) sm.pre[lo + i] = 0ull;
    sort_desc(sm.pre + lo, M);
    for (int r = lo + tid; r < hi; r += SB) {
      const DF e = df_exp2_rel(comp_value(sm.pre[r]), ctx, sm.e2h, sm.e2l);
      sm.esh[r] = e.h;
      sm.esl[r] = e.l;
    }
    __syncthreads();
    if (!topp) {  // top-k alone
      kept = nv;
      break;
    }
    if (!full) {
      // Z over the top-k survivors (all in this first and only block)
      DF acc = {0.0f, 0.0f};
      for (int r = tid; r < nv; r += SB) df_accumulate(acc, DF{sm.esh[r], sm.esl[r]});
      pz = df_mul_f(block_sum_df(df_fast_two_sum(acc.h, acc.l), sm), P.top_p);
    }
    if (tid < 32) {
      int k;
      const bool c = topp_scan_warp(sm.esh + lo, sm.esl + lo, M, lo, carry, pz, &k);
      if (tid == 0) {
        sm.done = (c || hi == nv) ? 1 : 0;
        sm.kept = lo + k;
        // top-p over everything with its crossing past the extracted prefix
        sm.flag = (!c && hi == nv && full) ? 1 : 0;
      }
    }
    __syncthreads();
    const bool done = sm.done != 0;
    kept = sm.kept;
    fallback = sm.flag != 0;
    __syncthreads();
    if (done) break;
    lo = hi;
    upper = cut;
    blk *= 2;
  }
  if (!fallback) {
    // the prefix the decision read: the kept set, and for top-k the K
    // survivors Z sums over.  A chunk that holds more tokens than it gave
    // can hide one inside it only if its last candidate lies strictly inside.
    const uint64_t last = sm.pre[(full ? kept : nv) - 1];
    if (tid == 0) sm.flag = 0;
    __syncthreads();
    if (tid < nch) {
      const int chunk_tokens = min(CHUNK, V - tid * CHUNK);
      if (chunk_tokens > nc && recs[tid].cand[nc - 1] > last) sm.flag = 1;
    }
    __syncthreads();
    fallback = sm.flag != 0;
    __syncthreads();
  }
  if (fallback) return general_sample(row, V, P, top1, sm);
  auto pget = [&](int r) { return sm.pre[r]; };
  return gumbel_pick(P, kept, pget, sm.esh, sm);
}

// ---------------------------------------------------------------------------
// row parameters
// ---------------------------------------------------------------------------
__device__ __forceinline__ RowParams row_params(int V, uint64_t seed, int64_t step, float temp,
                                                int32_t top_k, float top_p, uint32_t salt) {
  RowParams P;
  P.temperature = temp;
  P.top_k = top_k;
  P.top_p = top_p;
  P.salt = salt;
  P.seed = seed;
  P.step = step;
  P.K = (top_k > 0 && top_k < V) ? top_k : V;
  if (!(temp > 1e-5f))
    P.mode = MODE_GREEDY;
  else if (P.K <= MAXK_FAST)
    P.mode = MODE_TOPK_SMALL;
  else if (P.K == V)
    P.mode = (top_p < 1.0f) ? MODE_TOPP_FULL : MODE_ALL;
  else
    P.mode = MODE_GENERAL;
  const int kcap = P.mode == MODE_TOPK_SMALL ? P.K : MAXK_FAST;
  const int nch = (V + CHUNK - 1) / CHUNK;
  const int spread = (kcap + nch - 1) / nch;
  P.nc = min(kcap, max(NCAND, spread));
  const DF c2 = P.mode == MODE_GREEDY ? DF{0.0f, 0.0f} : df_div_f(DF{LOG2E_H, LOG2E_L}, temp);
  P.c2h = c2.h;
  P.c2l = c2.l;
  return P;
}

__device__ __forceinline__ int32_t kind_of(int32_t tok, const int32_t *stop, int n_stop, int32_t lo,
                                           int32_t hi) {
  for (int i = 0; i < n_stop; ++i)
    if (__ldg(stop + i) == tok) return PKV_KIND_STOP;
  return (tok >= lo && tok < hi) ? PKV_KIND_AUDIO : PKV_KIND_OTHER;
}

struct SampleArgs {
  const float *logits;
  int64_t row_stride;
  int batch;
  int vocab;
  int nch;
  const int32_t *slots;
  const int32_t *active;
  int num_slots;
  const uint64_t *seeds;
  int64_t *steps;
  const float *temperature;
  const int32_t *top_k;
  const float *top_p;
  uint32_t salt;
  int advance;
  const int32_t *stop_tokens;
  int n_stop;
  int32_t audio_lo, audio_hi;
  int32_t *out_tok;
  int32_t *out_kind;
  ChunkRec *recs;  // [B][nch]
  int32_t *err;
};

__global__ void __launch_bounds__(SB) sample_chunk_kernel(const SampleArgs a) {
  __shared__ SampSmem sm;
  const int b = blockIdx.y;
  const int c = blockIdx.x;
  if (!a.active[b]) return;
  const int slot = a.slots[b];
  if (slot < 0 || slot >= a.num_slots) return;
  load_exp2_table(sm);
  const RowParams P = row_params(a.vocab, a.seeds[slot], a.steps[slot], a.temperature[slot],
                                 a.top_k[slot], a.top_p[slot], a.salt);
  chunk_pass(a.logits + (int64_t)b * a.row_stride, a.vocab, c, P, a.recs + (int64_t)b * a.nch + c,
             sm, a.err);
}

__global__ void __launch_bounds__(SB) sample_finish_kernel(const SampleArgs a) {
  __shared__ SampSmem sm;
  const int b = blockIdx.x;
  if (!a.active[b]) {
    if (threadIdx.x == 0) {
      a.out_tok[b] = 0;
      a.out_kind[b] = PKV_KIND_OTHER;
    }
    return;
  }
  const int slot = a.slots[b];
  if (slot < 0 || slot >= a.num_slots) {
    if (threadIdx.x == 0) {
      a.out_tok[b] = 0;
      a.out_kind[b] = PKV_KIND_OTHER;
      report(a.err, PKV_DEV_ERR_SLOT);
    }
    return;
  }
  load_exp2_table(sm);
  const RowParams P = row_params(a.vocab, a.seeds[slot], a.steps[slot], a.temperature[slot],
                                 a.top_k[slot], a.top_p[slot], a.salt);
  __syncthreads();
  const int tok = finish_row(a.logits + (int64_t)b * a.row_stride, a.vocab, a.nch, P,
                             a.recs + (int64_t)b * a.nch, sm);
  if (threadIdx.x == 0) {
    a.out_tok[b] = tok;
    a.out_kind[b] = kind_of(tok, a.stop_tokens, a.n_stop, a.audio_lo, a.audio_hi);
    if (a.advance) a.steps[slot] = P.step + 1;
  }
}

struct FrameArgs {
  const float *base;  // [n_cb][B][V]
  const float *fb;    // [n_cb][V][V] or null
  int n_cb;
  int batch;
  int vocab;
  int nch;
  const int32_t *slots;
  const int32_t *active;
  int num_slots;
  const uint64_t *seeds;
  int64_t *steps;
  const float *temperature;
  const int32_t *top_k;
  const float *top_p;
  int32_t *out_codes;
  int32_t *out_kind;
  ChunkRec *recs;   // [B][nch]
  float *rows;      // [B][V]
  int32_t *err;
};

__global__ void __launch_bounds__(SB) frame_kernel(const FrameArgs a) {
  __shared__ SampSmem sm;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int V = a.vocab;
  if (!a.active[b]) {
    for (int j = tid; j < a.n_cb; j += SB) a.out_codes[(int64_t)b * a.n_cb + j] = 0;
    if (tid == 0) a.out_kind[b] = PKV_KIND_OTHER;
    return;
  }
  const int slot = a.slots[b];
  if (slot < 0 || slot >= a.num_slots) {
    for (int j = tid; j < a.n_cb; j += SB) a.out_codes[(int64_t)b * a.n_cb + j] = 0;
    if (tid == 0) {
      a.out_kind[b] = PKV_KIND_OTHER;
      report(a.err, PKV_DEV_ERR_SLOT);
    }
    return;
  }
  load_exp2_table(sm);
  const int64_t step = a.steps[slot];
  ChunkRec *recs = a.recs + (int64_t)b * a.nch;
  float *rowbuf = a.rows + (int64_t)b * V;
  int prev = 0;
  for (int j = 0; j < a.n_cb; ++j) {
    const float *row = a.base + ((int64_t)j * a.batch + b) * V;
    if (j > 0 && a.fb != nullptr) {
      const float *f = a.fb + ((int64_t)j * V + prev) * V;
      for (int i = tid; i < V; i += SB) rowbuf[i] = __fadd_rn(row[i], f[i]);
      __syncthreads();
      row = rowbuf;
    }
    const RowParams P = row_params(V, a.seeds[slot], step, a.temperature[slot], a.top_k[slot],
                                   a.top_p[slot], (uint32_t)(1 + j));
    __syncthreads();
    for (int c = 0; c < a.nch; ++c) {
      chunk_pass(row, V, c, P, recs + c, sm, a.err);
      __syncthreads();
    }
    const int tok = finish_row(row, V, a.nch, P, recs, sm);
    if (tid == 0) {
      a.out_codes[(int64_t)b * a.n_cb + j] = tok;
      sm.token = tok;
    }
    __syncthreads();
    prev = min(max(sm.token, 0), V - 1);
    __syncthreads();
  }
  if (tid == 0) {
    a.out_kind[b] = PKV_KIND_AUDIO;
    a.steps[slot] = step + 1;
  }
}

static int chunks_for(int V) { return (V + CHUNK - 1) / CHUNK; }

}  // namespace pkv

extern "C" size_t pkv_sample_workspace_bytes(int batch, int vocab) {
  using namespace pkv;
  if (batch <= 0 || vocab <= 0) return 0;
  return align_up((size_t)batch * chunks_for(vocab) * sizeof(ChunkRec), 256);
}

extern "C" size_t pkv_frame_workspace_bytes(int n_codebooks, int batch, int vocab) {
  using namespace pkv;
  if (n_codebooks <= 0 || batch <= 0 || vocab <= 0) return 0;
  return align_up((size_t)batch * chunks_for(vocab) * sizeof(ChunkRec), 256) +
         align_up((size_t)batch * vocab * sizeof(float), 256);
}

static int check_sampler_common(int batch, int vocab, const int32_t *slots, const int32_t *active,
                                int num_slots, const uint64_t *seeds, const int64_t *steps,
                                const float *temperature, const int32_t *top_k,
                                const float *top_p) {
  if (batch <= 0 || vocab <= 0 || num_slots <= 0) return PKV_ERR_INVALID_ARG;
  if (!slots || !active || !seeds || !steps || !temperature || !top_k || !top_p)
    return PKV_ERR_INVALID_ARG;
  if (vocab > pkv::MAX_CHUNKS * pkv::CHUNK) return PKV_ERR_UNSUPPORTED;
  if (batch > 65535) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

extern "C" int pkv_seeded_sample(const float *logits, int64_t row_stride, int batch, int vocab,
                                 const int32_t *slots, const int32_t *active, int num_slots,
                                 const uint64_t *seeds, int64_t *steps, const float *temperature,
                                 const int32_t *top_k, const float *top_p, uint32_t salt,
                                 int advance, const int32_t *stop_tokens, int n_stop,
                                 int32_t audio_lo, int32_t audio_hi, int32_t *out_tok,
                                 int32_t *out_kind, void *workspace, size_t workspace_bytes,
                                 int32_t *err_word, void *stream) {
  using namespace pkv;
  int st = check_sampler_common(batch, vocab, slots, active, num_slots, seeds, steps, temperature,
                                top_k, top_p);
  if (st != PKV_OK) return st;
  if (!logits || !out_tok || !out_kind || row_stride < vocab) return PKV_ERR_INVALID_ARG;
  if (n_stop < 0 || (n_stop > 0 && !stop_tokens)) return PKV_ERR_INVALID_ARG;
  if (((uintptr_t)logits & 3u) != 0) return PKV_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < pkv_sample_workspace_bytes(batch, vocab))
    return PKV_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return PKV_ERR_INVALID_ARG;
  SampleArgs a;
  a.logits = logits;
  a.row_stride = row_stride;
  a.batch = batch;
  a.vocab = vocab;
  a.nch = chunks_for(vocab);
  a.slots = slots;
  a.active = active;
  a.num_slots = num_slots;
  a.seeds = seeds;
  a.steps = steps;
  a.temperature = temperature;
  a.top_k = top_k;
  a.top_p = top_p;
  a.salt = salt;
  a.advance = advance != 0;
  a.stop_tokens = stop_tokens;
  a.n_stop = n_stop;
  a.audio_lo = audio_lo;
  a.audio_hi = audio_hi;
  a.out_tok = out_tok;
  a.out_kind = out_kind;
  a.recs = static_cast<ChunkRec *>(workspace);
  a.err = err_word;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  sample_chunk_kernel<<<dim3((unsigned)a.nch, (unsigned)batch), SB, 0, s>>>(a);
  int rc = launch_status();
  if (rc != PKV_OK) return rc;
  sample_finish_kernel<<<(unsigned)batch, SB, 0, s>>>(a);
  return launch_status();
}

extern "C" int pkv_codebook_frame_sample(const float *base, const float *fb, int n_codebooks,
                                         int batch, int vocab, const int32_t *slots,
                                         const int32_t *active, int num_slots,
                                         const uint64_t *seeds, int64_t *steps,
                                         const float *temperature, const int32_t *top_k,
                                         const float *top_p, int32_t *out_codes,
                                         int32_t *out_kind, void *workspace,
                                         size_t workspace_bytes, int32_t *err_word,
                                         void *stream) {
  using namespace pkv;
  int st = check_sampler_common(batch, vocab, slots, active, num_slots, seeds, steps, temperature,
                                top_k, top_p);
  if (st != PKV_OK) return st;
  if (!base || !out_codes || !out_kind || n_codebooks <= 0) return PKV_ERR_INVALID_ARG;
  if (((uintptr_t)base & 3u) != 0 || ((uintptr_t)fb & 3u) != 0) return PKV_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < pkv_frame_workspace_bytes(n_codebooks, batch, vocab))
    return PKV_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return PKV_ERR_INVALID_ARG;
  FrameArgs a;
  a.base = base;
  a.fb = fb;
  a.n_cb = n_codebooks;
  a.batch = batch;
  a.vocab = vocab;
  a.nch = chunks_for(vocab);
  a.slots = slots;
  a.active = active;
  a.num_slots = num_slots;
  a.seeds = seeds;
  a.steps = steps;
  a.temperature = temperature;
  a.top_k = top_k;
  a.top_p = top_p;
  a.out_codes = out_codes;
  a.out_kind = out_kind;
  a.recs = static_cast<ChunkRec *>(workspace);
  a.rows = reinterpret_cast<float *>(static_cast<unsigned char *>(workspace) +
                                     align_up((size_t)batch * a.nch * sizeof(ChunkRec), 256));
  a.err = err_word;
  frame_kernel<<<(unsigned)batch, SB, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return launch_status();
}
