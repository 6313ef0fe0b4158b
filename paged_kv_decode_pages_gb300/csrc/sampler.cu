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
// its own logits and slot state only.  Every decision (order, top-p cut,
// Gumbel argmax) is taken in fp64; the values compared are exact functions
// of the fp32 logits except the top-p normaliser's chunk partials, which
// are within 3e-9 of themselves (see the chunk pass).
//
// Structure:
//  * order key: the fp32 logit mapped to a uint32 that sorts like the float
//    (-0 folded onto +0); composite = key << 32 | ~token, so a larger
//    composite comes first in (value desc, id asc) order, and composites
//    are unique.
//  * chunk pass (one CTA per 8192-token chunk of a row; its logits are
//    loaded before the row's settings): chunk maximum; the chunk's nc
//    largest composites, nc = min(kcap, max(64, ceil(kcap / chunks))) with
//    kcap = the top-k, or 512 for top-p over the whole vocabulary, and the
//    smallest of them.  For nc <= 256 they come from a lower bound taken
//    from the warps' sorted thread maxima and exact rank counting over the
//    few composites above it (block_top_n), in descending order; otherwise,
//    or when more than 256 composites pass the bound, from a radix select
//    over 8-bit digits;
//    for top-p over the whole vocabulary, the partial normaliser
//    sum exp(x - x_chunkmax) = sum 2^(logit * log2(e) / T - t_chunkmax) in
//    double-float arithmetic (fp32 pairs): Tang's table-driven exp2 (ACM
//    TOMS 15(2), 1989) with a double-float table of 2^(j/32) and a degree-4
//    polynomial, each term within 3e-9 of itself, summed with exact
//    two-sum corrections -- on this GPU one fp64 warp instruction costs as
//    much issue time as several dozen fp32 ones, and this is the only
//    per-logit transcendental of the path; for "keep everything", the
//    chunk's Gumbel argmax.  The chunking depends on the vocabulary only.
//  * finish (one CTA per row): the kcap largest of the chunks' candidates,
//    in order (block_top_n over the union when kcap <= 256, else a radix
//    select over the union and a bitonic sort); top-k / top-p with fp64 prefix
//    sums in sorted order (a warp prefix scan, exponentials computed in
//    blocks only as far as the scan reaches); the Gumbel argmax.  The
//    sorted candidates are the exact global order over the prefix the
//    decision read unless a chunk holding more tokens than it gave has its
//    smallest candidate strictly inside that prefix; such rows, and rows
//    whose kept set is not decided by kcap tokens (top-k > 512, or top-p
//    needing more than 512 tokens), take an exact general path that streams
//    the row: radix select of the top-k threshold and progressive sorted
//    extraction until the top-p crossing.
//  * further settings (pkv_seeded_sample_ext; "Adding a Model", "2. The
//    program", in the order of the Chatterbox notes of "Supported Models"
//    with top-k before min_p): the repetition penalty is applied to the
//    order keys of the window's tokens as the chunk pass loads them (a
//    shared bitmap per chunk, copied to the workspace for the general
//    path); min_p cuts the sorted candidates at the first rank >= 1 with
//    exp(x - x_max) < min_p and top-p renormalises over the ranks before
//    it; the raw log-prob uses per-chunk log-sum-exp partials of the
//    unprocessed logits, the processed one the kept ranks' mass.
//  * the frame kernel runs the same chunk pass and finish for each of the
//    codebooks in turn inside one CTA per row.
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int SB = 256;                 // threads per sampler CTA
constexpr int CHUNK = 8192;             // tokens per chunk
constexpr int EPT = CHUNK / SB;         // tokens per thread in a chunk pass
constexpr int NCAND = 512;              // most candidates kept per chunk
constexpr int NC_MIN = 64;              // least candidates kept per chunk
constexpr int MAX_CHUNKS = 64;          // vocab <= 64 * 8192
constexpr int GEN_BLOCK = 1024;         // sorted block (finish and general path)

enum Mode : int { MODE_GREEDY = 0, MODE_TOPK_SMALL = 1, MODE_TOPP_FULL = 2, MODE_ALL = 3, MODE_GENERAL = 4 };

struct ChunkRec {
  uint64_t top1;       // largest composite of the chunk (0: chunk empty)
  uint64_t thr;        // the smallest of them when the chunk holds more tokens (else 0)
  double gscore;       // best x + g of the chunk                  (MODE_ALL)
  int32_t gid;         // its token
  int32_t ncand;       // candidates kept
  float zh, zl;        // sum over the chunk of 2^(t - t_top1), double-float  (need_z)
  float rmax;          // largest unprocessed logit of the chunk      (raw log-probs)
  float rzh, rzl;      // sum over the chunk of exp(logit - rmax)      (raw log-probs)
  uint32_t gkey;       // order key of gid                            (MODE_ALL)
  uint64_t pad_;
  uint64_t cand[NCAND];
};
static_assert(sizeof(ChunkRec) % 64 == 0, "ChunkRec");

struct RowParams {
  float temperature;
  int32_t top_k;
  float top_p;
  uint32_t salt;
  uint64_t seed;
  int64_t step;
  int K;       // top-k count after normalisation (V when off)
  int mode;
  int nc;      // candidates per chunk
  float c2h, c2l;  // log2(e) / T as a double-float
  // further controls (pkv_seeded_sample_ext; all off otherwise)
  float min_p;           // <= 0: off
  float pen;             // repetition penalty
  int n_pen;             // window length (0: no penalty)
  const int32_t *hist;   // the slot's ring of sampled tokens
  int64_t hist_len;
  int hist_cap;
  int lp_raw, lp_proc;   // log-probs requested
  int need_z;            // chunk pass computes the normaliser over the whole row
};

// i-th newest token of the penalty window
__device__ __forceinline__ int32_t pen_token(const RowParams &P, int i) {
  return P.hist[(P.hist_len - 1 - i) % P.hist_cap];
}

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

__device__ __forceinline__ Exp2Ctx exp2_ctx(float c2h, float c2l, float vmax) {
  const DF tm = df_mul_f(DF{c2h, c2l}, vmax);
  return {c2h, c2l, tm.h, tm.l};
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

__device__ __forceinline__ double gumbel(const RowParams &P, int token) {
  const uint64_t w = philox_word0(P.seed, P.salt, (uint64_t)(uint32_t)token, (uint64_t)P.step);
  const double u = (double)(2ull * (w >> 12) + 1ull) * 0x1p-53;
  return -log(-log(u));
}

constexpr float LN2F = 0.693147180559945309f;

// The same noise in fp32, for screening only: within ~1e-5 absolute of the
// fp64 value (see finish_row's margin).  E = -ln(u) is formed without
// cancellation: for u < 1/2 from u itself (relative error 2^-24 in u), for
// u >= 1/2 from v = 1 - u = (2^53 - 2j - 1) 2^-53, which is exact as an
// integer, by the series v + v^2/2 + ... + v^8/8 when v < 1/8 (the rest is
// below 1e-9 v) and by ln(1 - v) otherwise (then E > 0.13).
__device__ __forceinline__ float gumbel32(const RowParams &P, int token) {
  const uint64_t w = philox_word0(P.seed, P.salt, (uint64_t)(uint32_t)token, (uint64_t)P.step);
  const uint64_t j = w >> 12;
  float e;
  if (j < (1ull << 51)) {
    e = -lg2_approx(__ull2float_rn(2ull * j + 1ull) * 0x1p-53f) * LN2F;
  } else {
    const float v = __ull2float_rn((1ull << 53) - 2ull * j - 1ull) * 0x1p-53f;
    if (v < 0.125f) {
      float q = 1.0f / 8.0f;
      q = fmaf(q, v, 1.0f / 7.0f);
      q = fmaf(q, v, 1.0f / 6.0f);
      q = fmaf(q, v, 1.0f / 5.0f);
      q = fmaf(q, v, 1.0f / 4.0f);
      q = fmaf(q, v, 1.0f / 3.0f);
      q = fmaf(q, v, 1.0f / 2.0f);
      q = fmaf(q, v, 1.0f);
      e = q * v;
    } else {
      e = -lg2_approx(1.0f - v) * LN2F;
    }
  }
  return -lg2_approx(e) * LN2F;
}

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
__device__ __forceinline__ double comp_x(uint64_t c, float temperature) {
  return (double)key_value((uint32_t)(c >> 32)) / (double)temperature;
}

// repetition penalty of one logit: a positive logit is divided by the
// penalty, any other multiplied by it (fp32, correctly rounded)
__device__ __forceinline__ float penalise(float v, float pen) {
  return v > 0.0f ? __fdiv_rn(v, pen) : __fmul_rn(v, pen);
}

// A logits row as the sampler sees it: the fp32 values with the penalty
// applied to the tokens marked in pbits (one bit per token; null: none).
struct RowView {
  const float *x;
  const uint32_t *pbits;
  float pen;
  __device__ __forceinline__ uint32_t key(int i, bool &bad) const {
    float v = x[i];
    if (pbits != nullptr && ((pbits[i >> 5] >> (i & 31)) & 1u)) v = penalise(v, pen);
    return order_key(v, bad);
  }
};

// ---------------------------------------------------------------------------
// shared scratch
// ---------------------------------------------------------------------------
struct SampSmem {
  float e2h[32], e2l[32];  // the 2^(j/32) table
  float wh[SB / 32], wl[SB / 32];
  uint32_t hist[256];
  uint64_t red_u64[SB / 32];
  uint64_t red_u64b[SB / 32];
  double red_d[SB];
  int32_t red_i[SB];
  uint64_t sel_prefix;
  uint32_t sel_want;
  uint32_t sel_done;
  uint32_t cnt;
  int32_t flag;
  int32_t token;
  int32_t kept;
  int32_t done;
  int32_t kp;
  double zsum;
  double s_kept;     // mass (relative to the row maximum) of the kept tokens
  double m_row;      // x of the row maximum
  double xbest;      // x of the sampled token
  uint32_t penbits[CHUNK / 32];  // penalised tokens of the chunk
  uint64_t sortbuf[GEN_BLOCK];
  double es[GEN_BLOCK];
  uint64_t gbuf[SB];             // block_top_n's gather buffer (finish)
  float eh[NCAND], el[NCAND];    // 2^(t_r - t_0) of the sorted candidates, double-float
  float g32[NCAND];              // their fp32 Gumbel noise
  float s32[NCAND];              // their fp32 scores
  float fh[MAX_CHUNKS], fl[MAX_CHUNKS];  // the chunks' rescaled normalisers
  float wbs[SB / 32];            // per-warp best fp32 scores
  float zh, zl;                  // a normaliser, double-float
};

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
  for (int w = 1; w < SB / 32; ++w) r = sm.red_u64[w] > r ? sm.red_u64[w] : r;
  __syncthreads();
  return r;
}

// Sum in a fixed order: thread partials, then a fixed binary tree.
__device__ double block_sum_d(double v, SampSmem &sm) {
  __syncthreads();
  sm.red_d[threadIdx.x] = v;
  __syncthreads();
  for (int s = SB / 2; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) sm.red_d[threadIdx.x] += sm.red_d[threadIdx.x + s];
    __syncthreads();
  }
  const double r = sm.red_d[0];
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
  for (int w = 1; w < SB / 32; ++w) r = df_add(r, DF{sm.wh[w], sm.wl[w]});
  __syncthreads();
  return r;
}

__device__ __forceinline__ void load_exp2_table(SampSmem &sm) {
  if (threadIdx.x < 32) {
    sm.e2h[threadIdx.x] = c_exp2_tab_h[threadIdx.x];
    sm.e2l[threadIdx.x] = c_exp2_tab_l[threadIdx.x];
  }
}

// Argmax of (score desc, id asc); ids < 0 mark "none".
__device__ __forceinline__ bool better(double s, int id, double bs, int bid) {
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

// Bitonic sort of n (power of two) u64 values in shared memory, descending.
__device__ void block_sort_desc(uint64_t *v, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      // one compare-exchange pair (i, i + j) per thread, bit j of i clear
      for (int p = threadIdx.x; p < n / 2; p += SB) {
        const int i = ((p & ~(j - 1)) << 1) | (p & (j - 1));
        const uint64_t a = v[i], b = v[i + j];
        const bool desc_block = (i & k) == 0;
        if (desc_block ? (a < b) : (a > b)) {
          v[i] = b;
          v[i + j] = a;
        }
      }
      __syncthreads();
    }
  }
}

// Warp 0 walks the 256-bin histogram from the top bin down and picks the
// bin holding the `want`-th (1-based) largest element.  Results in sm.
__device__ void select_bin(SampSmem &sm, int shift) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    // lane covers bins 255-8*lane .. 248-8*lane (descending)
    // every lane reads the wanted rank before the scan below (a warp-wide
    // sync point), as one lane overwrites it afterwards
    const uint32_t want = sm.sel_want;
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

// ---------------------------------------------------------------------------
// chunk pass
// ---------------------------------------------------------------------------
// The per-logit loops below with a long body (the double-float exponential,
// the fp64 Gumbel noise) are rolled loops over the chunk as it lies in global
// memory (just loaded, so served from L1 / L2): unrolled over the thread's
// 32 values they were tens of kilobytes of straight-line code, executed once
// per CTA and stalled on instruction fetch.

// Sum over the chunk's logits v (penalised where the chunk's bitmap in
// sm.penbits says so, when pen_on) of 2^(v * c2 - t_max), in double-float;
// all threads get it.  NaN and -inf logits add 0.
__device__ __forceinline__ DF chunk_exp_sum(const float *row, int start, int cnt, const Exp2Ctx ctx,
                                         bool pen_on, float pen, SampSmem &sm) {
  DF acc = {0.0f, 0.0f};
#pragma unroll 2
  for (int i = (int)threadIdx.x; i < cnt; i += SB) {
    float v = row[start + i];
    if (pen_on && ((sm.penbits[i >> 5] >> (i & 31)) & 1u)) v = penalise(v, pen);
    if (v == 0.0f) v = 0.0f;  // -0 ranks as +0
    df_accumulate(acc, df_exp2_rel(v, ctx, sm.e2h, sm.e2l));
  }
  return block_sum_df(df_fast_two_sum(acc.h, acc.l), sm);
}

// Keep everything: the thread's best x + g (fp64, the definition) over the
// chunk's tokens; *bid < 0 when the thread has none.
__device__ __forceinline__ void chunk_gumbel_all(const float *row, int start, int cnt,
                                              const RowParams P, SampSmem &sm, double *bs,
                                              int *bid, uint32_t *bkey) {
  *bs = 0.0;
  *bid = -1;
  *bkey = 0u;
  const bool pen_on = P.n_pen > 0;
#pragma unroll 1
  for (int i = (int)threadIdx.x; i < cnt; i += SB) {
    float v = row[start + i];
    if (pen_on && ((sm.penbits[i >> 5] >> (i & 31)) & 1u)) v = penalise(v, P.pen);
    bool bad = false;
    const uint32_t key = order_key(v, bad);
    const int tok = start + i;
    const double s = (double)key_value(key) / (double)P.temperature + gumbel(P, tok);
    if (better(s, tok, *bs, *bid)) {
      *bs = s;
      *bid = tok;
      *bkey = key;
    }
  }
}

// The largest of a thread's N values get(j), as four independent partial
// maxima (short dependency chains)
template <int N, class Get>
__device__ __forceinline__ uint64_t thread_max(Get get) {
  uint64_t m[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const uint64_t x = get(j);
    m[j & 3] = x > m[j & 3] ? x : m[j & 3];
  }
  const uint64_t a = m[0] > m[1] ? m[0] : m[1], b = m[2] > m[3] ? m[2] : m[3];
  return a > b ? a : b;
}

// The n largest of the block's values without a radix select or a full
// sort.  Each thread holds N values, get(j) for j < N; 0 means "no value" and
// the other values are distinct.  Needs n <= SB and at least n nonzero
// values.  A lower bound L with at least n values >= L comes from the
// threads' largest values: each warp sorts its 32 (a bitonic network over
// the lanes) and offers its q-th largest, q = ceil(n / 8); L is the
// smallest offer, so every warp holds q values >= L (or L is 0 and every
// nonzero value passes).  The nonzero values >= L -- typically a few dozen
// more than n -- are gathered into gbuf (SB entries, shared memory) and
// each one's rank among them is counted: ranks 0 .. n-1 are the n largest,
// written to out[rank] (descending order), and rank n-1 also to *thr when
// thr is not null.  top1 receives the largest value in any case.  Returns
// false, having written nothing to out, when more than SB values pass the
// bound.
template <int N, class Get>
__device__ bool block_top_n(Get get, int n, uint64_t *out, uint64_t *thr, uint64_t *gbuf,
                            SampSmem &sm, uint64_t &top1) {
  constexpr int NW = SB / 32;
  static_assert(N <= 32, "N");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = (n + NW - 1) / NW;
  uint64_t v = thread_max<N>(get);
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t o = __shfl_xor_sync(FULL_MASK, v, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
      v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  const uint64_t offer = __shfl_sync(FULL_MASK, v, q - 1);
  __syncthreads();  // earlier readers of red_u64, red_u64b, cnt and gbuf are done
  if (lane == 0) {
    sm.red_u64[warp] = offer;
    sm.red_u64b[warp] = v;  // the warp's largest
  }
  if (tid == 0) sm.cnt = 0;
  __syncthreads();
  uint64_t L = sm.red_u64[0], top = sm.red_u64b[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) {
    L = sm.red_u64[w] < L ? sm.red_u64[w] : L;
    top = sm.red_u64b[w] > top ? sm.red_u64b[w] : top;
  }
  top1 = top;
  // gather: a slot range per warp (one atomic), lanes in order inside it;
  // bit j of pm marks the thread's value j (independent tests, no chain)
  uint32_t pm = 0;
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const uint64_t x = get(j);
    if (x != 0ull && x >= L) pm |= 1u << j;
  }
  const int cnt = __popc(pm);
  int incl = cnt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(FULL_MASK, incl, off);
    if (lane >= off) incl += t;
  }
  int base = 0;
  if (lane == 31) base = (int)atomicAdd(&sm.cnt, (uint32_t)incl);
  base = __shfl_sync(FULL_MASK, base, 31);
  const int pos = base + incl - cnt;
#pragma unroll
  for (int j = 0; j < N; ++j)
    if ((pm >> j) & 1u) {
      const int at = pos + __popc(pm & ((1u << j) - 1u));
      if (at < SB) gbuf[at] = get(j);
    }
  __syncthreads();
  const int C = (int)sm.cnt;
  if (C > SB) return false;  // the same answer in every thread
  if (tid < C) {
    const uint64_t me = gbuf[tid];
    int r = 0;
    for (int k = 0; k < C; ++k) r += gbuf[k] > me ? 1 : 0;
    if (r < n) out[r] = me;
    if (r == n - 1 && thr != nullptr) *thr = me;
  }
  __syncthreads();
  return true;
}

// The thread's logits of chunk c (element tid + j * SB in raw[j]), every
// load issued before any is used so that all of them are in flight at once.
// The frame kernel writes the rows it samples: plain loads, no __ldg.
__device__ __forceinline__ void load_chunk(const float *row, int V, int c, float (&raw)[EPT]) {
  const int tid = threadIdx.x;
  const int start = c * CHUNK;
  const int cnt = min(CHUNK, V - start);
  if (cnt == CHUNK) {
#pragma unroll
    for (int j = 0; j < EPT; ++j) raw[j] = row[start + tid + j * SB];
  } else {
#pragma unroll
    for (int j = 0; j < EPT; ++j) raw[j] = tid + j * SB < cnt ? row[start + tid + j * SB] : 0.0f;
  }
}

// raw: the thread's logits of chunk c (load_chunk).  pbits: the row's
// penalty bitmap in global memory, written for this chunk when the row is
// penalised (may be null otherwise)
__device__ void chunk_pass(const float (&raw)[EPT], const float *row, int V, int c,
                           const RowParams &P, ChunkRec *rec, uint32_t *pbits, SampSmem &sm,
                           int32_t *err) {
  const int tid = threadIdx.x;
  const int start = c * CHUNK;
  const int cnt = min(CHUNK, V - start);
  uint32_t key[EPT];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int i = tid + j * SB;
    key[j] = (i < cnt) ? order_key(raw[j], bad) : 0u;
  }
  if (bad) report(err, PKV_DEV_ERR_LOGITS);
  if (P.lp_raw) {
    // raw log-softmax partials: chunk maximum of the unprocessed logits and
    // sum exp(logit - max) = sum 2^((logit - max) log2(e))
    uint32_t km = 0;
#pragma unroll
    for (int j = 0; j < EPT; ++j)
      if (tid + j * SB < cnt) km = key[j] > km ? key[j] : km;
    const float rmax = key_value((uint32_t)block_max_u64(km, sm));
    const DF z = chunk_exp_sum(row, start, cnt, exp2_ctx(LOG2E_H, LOG2E_L, rmax), false, 1.0f,
                               sm);
    if (tid == 0) {
      rec->rmax = rmax;
      rec->rzh = z.h;
      rec->rzl = z.l;
    }
  }
  if (P.n_pen > 0) {
    // the penalty window's tokens that fall in this chunk, as a bitmap
    // (a token repeated in the window is penalised once)
    for (int w = tid; w < CHUNK / 32; w += SB) sm.penbits[w] = 0u;
    __syncthreads();
    for (int i = tid; i < P.n_pen; i += SB) {
      const int32_t t = pen_token(P, i);
      if (t >= start && t < start + cnt)
        atomicOr(&sm.penbits[(t - start) >> 5], 1u << ((t - start) & 31));
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int i = tid + j * SB;
      if (i < cnt && ((sm.penbits[i >> 5] >> (i & 31)) & 1u)) {
        bool b2 = false;
        key[j] = order_key(penalise(key_value(key[j]), P.pen), b2);
      }
    }
    if (pbits != nullptr)
      for (int w = tid; w < (cnt + 31) / 32; w += SB) pbits[c * (CHUNK / 32) + w] = sm.penbits[w];
  }
  auto comp_at = [&](int j) -> uint64_t {
    const int i = tid + j * SB;
    return i < cnt ? composite(key[j], start + i) : 0ull;
  };
  // the chunk's nc largest composites (candidate modes), and its largest
  const int nc = P.nc;
  const bool sel = P.mode == MODE_TOPK_SMALL || P.mode == MODE_TOPP_FULL;
  uint64_t top1 = 0;
  bool fast = false;
  if (sel && cnt > nc && nc <= SB) {
    fast = block_top_n<EPT>(comp_at, nc, rec->cand, &rec->thr, sm.sortbuf, sm, top1);
    if (fast && tid == 0) rec->ncand = nc;
  } else {
    top1 = block_max_u64(thread_max<EPT>(comp_at), sm);
  }
  if (tid == 0) rec->top1 = top1;
  if (P.mode == MODE_GREEDY || P.mode == MODE_GENERAL) return;

  if (P.mode == MODE_ALL) {
    double bs;
    int bid;
    uint32_t bkey;
    chunk_gumbel_all(row, start, cnt, P, sm, &bs, &bid, &bkey);
    double best;
    const int id = block_argmax(bs, bid, sm, &best);
    if (tid == 0) {
      rec->gscore = best;
      rec->gid = id;
    }
    if (bid == id && id >= 0) rec->gkey = bkey;
  } else {
    // the chunk's nc largest composites, unless the fast selection wrote them
    uint64_t thr = 0;  // keep composites >= thr
    if (!fast && cnt > nc) {
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
    if (!fast) {
      if (tid == 0) sm.cnt = 0;
      __syncthreads();
#pragma unroll
      for (int j = 0; j < EPT; ++j) {
        const int i = tid + j * SB;
        if (i < cnt) {
          const uint64_t cc = composite(key[j], start + i);
          if (cc >= thr) {
            const uint32_t pos = atomicAdd(&sm.cnt, 1u);
            if (pos < (uint32_t)nc) rec->cand[pos] = cc;
          }
        }
      }
      __syncthreads();
      const int got = min((int)sm.cnt, nc);
      for (int i = got + tid; i < nc; i += SB) rec->cand[i] = 0;
      if (tid == 0) {
        rec->ncand = got;
        rec->thr = cnt > nc ? thr : 0ull;
      }
    }
  }

  if (P.need_z) {
    // sum over the chunk of exp(x - mx) = 2^(t - t_max), t = logit * log2(e) / T
    const Exp2Ctx ctx = exp2_ctx(P.c2h, P.c2l, key_value((uint32_t)(top1 >> 32)));
    const DF z = chunk_exp_sum(row, start, cnt, ctx, P.n_pen > 0, P.pen, sm);
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
// Composite of rank `rank` (0-based, descending) among the values get(i),
// i < n, that are below `upper` (0 marks "no value").  Requires that many
// such values to exist.
template <class Get>
__device__ uint64_t select_rank_of(int n, Get get, uint64_t upper, int rank, SampSmem &sm) {
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

// Composite of rank `rank` (0-based, descending) among elements with
// composite < upper.  Requires that many such elements to exist.
__device__ uint64_t select_rank(const RowView &rv, int V, uint64_t upper, int rank,
                                SampSmem &sm) {
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
    bool dummy = false;
    for (int i = threadIdx.x; i < V; i += SB) {
      const uint64_t cc = composite(rv.key(i, dummy), i);
      if (cc < upper && (cc & mask) == prefix) atomicAdd(&sm.hist[(cc >> shift) & 255u], 1u);
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

// z_known >= 0: the normaliser over the top-k survivors, already computed
// relative to the row maximum (top-p over the whole vocabulary, min_p off).
// With log-probs requested, leaves the kept mass, the row maximum's x and
// the sampled token's x in sm.s_kept, sm.m_row and sm.xbest.
__device__ int general_sample(const RowView &rv, int V, const RowParams &P, uint64_t top1,
                              double z_known, SampSmem &sm) {
  const int tid = threadIdx.x;
  const int K = P.K;
  const uint64_t thrK = (K < V) ? select_rank(rv, V, ~0ull, K - 1, sm) : 0ull;
  const double m = comp_x(top1, P.temperature);
  const bool minp = P.min_p > 0.0f;
  const bool topp = P.top_p < 1.0f;
  bool dummy = false;
  uint64_t thr = thrK;
  double S = 0.0;  // top-p: the kept mass
  if (topp) {
    double z = z_known;
    if (z < 0.0) {
      // the normaliser over the top-k survivors that pass min_p
      z = 0.0;
      for (int i = tid; i < V; i += SB) {
        const uint32_t key = rv.key(i, dummy);
        const uint64_t cc = composite(key, i);
        if (cc >= thrK) {
          const double e = exp((double)key_value(key) / (double)P.temperature - m);
          if (!minp || cc == top1 || e >= (double)P.min_p) z += e;
        }
      }
      z = block_sum_d(z, sm);
    }
    const double pz = (double)P.top_p * z;
    // progressive sorted extraction until the running sum reaches p * Z or
    // a token falls below min_p
    uint64_t upper = ~0ull;
    int taken = 0;
    uint64_t cutoff = top1;
    bool done = false;
    while (!done) {
      const int M = min(GEN_BLOCK, K - taken);
      const uint64_t lo = select_rank(rv, V, upper, M - 1, sm);
      if (tid == 0) sm.cnt = 0;
      __syncthreads();
      for (int i = tid; i < V; i += SB) {
        const uint64_t cc = composite(rv.key(i, dummy), i);
        if (cc >= lo && cc < upper) {
          const uint32_t pos = atomicAdd(&sm.cnt, 1u);
          if (pos < GEN_BLOCK) sm.sortbuf[pos] = cc;
        }
      }
      __syncthreads();
      int n2 = 1;
      while (n2 < M) n2 <<= 1;
      for (int i = M + tid; i < n2; i += SB) sm.sortbuf[i] = 0;
      __syncthreads();
      block_sort_desc(sm.sortbuf, n2);
      for (int r = tid; r < M; r += SB) sm.es[r] = exp(comp_x(sm.sortbuf[r], P.temperature) - m);
      __syncthreads();
      if (tid == 0) {
        int r = 0;
        for (; r < M; ++r) {
          if (taken + r == 0 || (S < pz && (!minp || sm.es[r] >= (double)P.min_p))) {
            S += sm.es[r];
            cutoff = sm.sortbuf[r];
          } else {
            break;
          }
        }
        sm.flag = (r < M || taken + M >= K) ? 1 : 0;
        sm.zsum = S;
        sm.sel_prefix = cutoff;
      }
      __syncthreads();
      done = sm.flag != 0;
      S = sm.zsum;
      cutoff = sm.sel_prefix;
      taken += M;
      upper = lo;
      __syncthreads();
    }
    thr = cutoff;
  }
  // Gumbel argmax over the kept tokens (composite >= thr; without top-p,
  // also passing min_p)
  const bool filt = minp && !topp;
  const bool mass = P.lp_proc && !topp;
  double bs = 0.0, bx = 0.0, sk = 0.0;
  int bid = -1;
  for (int i = tid; i < V; i += SB) {
    const uint32_t key = rv.key(i, dummy);
    const uint64_t cc = composite(key, i);
    if (cc >= thr) {
      const double x = (double)key_value(key) / (double)P.temperature;
      if (filt || mass) {
        const double e = exp(x - m);
        if (filt && !(cc == top1 || e >= (double)P.min_p)) continue;
        sk += e;
      }
      const double s = x + gumbel(P, i);
      if (better(s, i, bs, bid)) {
        bs = s;
        bid = i;
        bx = x;
      }
    }
  }
  const int id = block_argmax(bs, bid, sm);
  if (P.lp_proc) {
    const double kept_mass = topp ? S : block_sum_d(sk, sm);
    if (bid == id) sm.xbest = bx;
    if (tid == 0) {
      sm.s_kept = kept_mass;
      sm.m_row = m;
    }
    __syncthreads();
  }
  return id;
}

// ---------------------------------------------------------------------------
// finish: one CTA per row
// ---------------------------------------------------------------------------
// Arithmetic of the decision.  The definition is stated in fp64 (x = logit
// / T, e^(x - m), prefix sums against p * Z, x + Gumbel noise).  One fp64
// warp instruction costs this GPU as much issue time as several dozen fp32
// ones, and an fp64 logarithm thousands of cycles, so the finish works in
// double-float arithmetic and takes fp64 only where a decision could
// otherwise differ from the definition:
//  * e^(x_r - m) = 2^(t_r - t_0) by df_exp2_rel (within 3e-9 of itself), the
//    normaliser and the top-p prefix sums as double-float sums, so a cut can
//    differ from the fp64 definition only where a prefix sum lies within
//    ~1e-8 of p * Z, or e_r within ~1e-8 of min_p (near-ties);
//  * Gumbel-max: every kept rank's score x + g is formed in fp32 (x by a
//    correctly rounded division, g by gumbel32; within 2e-5 + 2.5e-7 |score|
//    of the fp64 score).  When no other kept rank lies within
//    1e-4 + 2e-6 |best| of the best fp32 score the fp32 winner is the fp64
//    winner; otherwise the ranks within that margin are scored again in fp64
//    exactly as the definition states, and the token is theirs.

constexpr int UNION_PT = 8;               // union slots per thread in union_top_n
constexpr int UNION_MAX = UNION_PT * SB;  // largest union taken by union_top_n

// The n largest composites of the union of the chunks' candidates (chunk c
// holds nc slots, zero past its ncand), in descending order, into
// sm.sortbuf[0, n).  Needs nu = nch * nc <= UNION_MAX, n <= SB and n
// nonzero slots; false (nothing written) when more than SB slots pass the
// selection bound.
__device__ bool union_top_n(const ChunkRec *recs, int nc, int nu, int n, SampSmem &sm) {
  const uint64_t magic = ((1ull << 32) + (uint64_t)nc - 1ull) / (uint64_t)nc;  // i / nc, i < 2^16
  auto get = [&](int k) -> uint64_t {
    const int i = (int)threadIdx.x + k * SB;
    if (i >= nu) return 0ull;
    const int c = (int)(((uint64_t)i * magic) >> 32);
    return recs[c].cand[i - c * nc];
  };
  uint64_t t1;
  return block_top_n<UNION_PT>(get, n, sm.sortbuf, nullptr, sm.gbuf, sm, t1);
}

// The nv largest composites of the union in descending order into
// sm.sortbuf[0, nv) (nv <= NCAND): a radix select of the nv-th, the gather,
// a bitonic sort.
__device__ void union_sorted_slow(const ChunkRec *recs, int nc, int nu, int nv, SampSmem &sm) {
  const int tid = threadIdx.x;
  auto cand_at = [&](int i) -> uint64_t { return recs[i / nc].cand[i % nc]; };
  const uint64_t thr = select_rank_of(nu, cand_at, ~0ull, nv - 1, sm);
  if (tid == 0) sm.cnt = 0;
  __syncthreads();
  for (int i = tid; i < nu; i += SB) {
    const uint64_t cc = cand_at(i);
    if (cc != 0ull && cc >= thr) {
      const uint32_t pos = atomicAdd(&sm.cnt, 1u);
      if (pos < (uint32_t)nv) sm.sortbuf[pos] = cc;
    }
  }
  __syncthreads();
  int n2 = 1;
  while (n2 < nv) n2 <<= 1;
  for (int i = nv + tid; i < n2; i += SB) sm.sortbuf[i] = 0ull;
  __syncthreads();
  block_sort_desc(sm.sortbuf, n2);
}

// The normaliser of the whole row relative to its maximum: the chunks'
// partials z_c (relative to each chunk's maximum) times 2^(t_c - t_0),
// added in chunk order.
__device__ DF row_normaliser(const ChunkRec *recs, int nch, const Exp2Ctx &ctx, SampSmem &sm) {
  const int tid = threadIdx.x;
  __syncthreads();
  if (tid < nch) {
    DF f = {0.0f, 0.0f};
    if (recs[tid].top1 != 0ull) {
      const DF w = df_exp2_rel(key_value((uint32_t)(recs[tid].top1 >> 32)), ctx, sm.e2h, sm.e2l);
      f = df_mul(DF{recs[tid].zh, recs[tid].zl}, w);
    }
    sm.fh[tid] = f.h;
    sm.fl[tid] = f.l;
  }
  __syncthreads();
  if (tid == 0) {
    DF z = {0.0f, 0.0f};
    for (int c = 0; c < nch; ++c) z = df_add(z, DF{sm.fh[c], sm.fl[c]});
    sm.zh = z.h;
    sm.zl = z.l;
  }
  __syncthreads();
  const DF z = {sm.zh, sm.zl};
  __syncthreads();
  return z;
}

// Warp 0: the first rank r >= max(lo, 1) in [lo, hi) with e_r < min_p, or -1.
__device__ int minp_boundary_warp(const SampSmem &sm, int lo, int hi, float min_p) {
  for (int base = max(lo, 1); base < hi; base += 32) {
    const int r = base + (int)(threadIdx.x & 31);
    bool below = false;
    if (r < hi) below = sm.eh[r] < min_p || (sm.eh[r] == min_p && sm.el[r] < 0.0f);
    const unsigned bm = __ballot_sync(FULL_MASK, below);
    if (bm) return base + __ffs(bm) - 1;
  }
  return -1;
}

// Warp 0: top-p over ranks [0, n): rank r is kept iff r == 0 or the sum of
// the e's before it is below pz (double-float prefix sums, 32 ranks at a
// time by shuffles).  Returns the first rank not kept, or n.
__device__ int topp_cut_warp(const SampSmem &sm, int n, DF pz) {
  const int lane = threadIdx.x & 31;
  DF carry = {0.0f, 0.0f};
  for (int base = 0; base < n; base += 32) {
    const int r = base + lane;
    DF inc = r < n ? DF{sm.eh[r], sm.el[r]} : DF{0.0f, 0.0f};
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const DF o = df_shfl_up(inc, off);
      if (lane >= off) inc = df_add(inc, o);
    }
    DF ex = df_shfl_up(inc, 1);
    if (lane == 0) ex = DF{0.0f, 0.0f};
    const DF before = df_add(carry, ex);
    const bool stop = r < n && r > 0 && !df_lt(before, pz);
    const unsigned bm = __ballot_sync(FULL_MASK, stop);
    if (bm) return base + __ffs(bm) - 1;
    carry = df_add(carry, df_shfl(inc, 31));
  }
  return n;
}

// Gumbel-max over the kept ranks [0, kept) of sm.sortbuf, whose fp32 noise
// is in sm.g32: the fp32 screen, then fp64 scores for the contenders within
// the margin (see the arithmetic note above).  Returns the composite of the
// winner.
__device__ uint64_t gumbel_argmax_sorted(const RowParams &P, int kept, SampSmem &sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (kept == 1) return sm.sortbuf[0];
  float bs = -INFINITY;
  uint64_t bc = 0ull;
  for (int r = tid; r < kept; r += SB) {
    const uint64_t cc = sm.sortbuf[r];
    const float s = __fadd_rn(__fdiv_rn(key_value((uint32_t)(cc >> 32)), P.temperature), sm.g32[r]);
    sm.s32[r] = s;
    if (bc == 0ull || s > bs || (s == bs && comp_token(cc) < comp_token(bc))) {
      bs = s;
      bc = cc;
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float os = __shfl_xor_sync(FULL_MASK, bs, off);
    const uint64_t oc = __shfl_xor_sync(FULL_MASK, bc, off);
    if (oc != 0ull && (bc == 0ull || os > bs || (os == bs && comp_token(oc) < comp_token(bc)))) {
      bs = os;
      bc = oc;
    }
  }
  __syncthreads();
  if (lane == 0) {
    sm.wbs[warp] = bs;
    sm.red_u64[warp] = bc;
  }
  __syncthreads();
  float best = -INFINITY;
  uint64_t bestc = 0ull;
  for (int w = 0; w < SB / 32; ++w) {
    const uint64_t oc = sm.red_u64[w];
    const float os = sm.wbs[w];
    if (oc != 0ull && (bestc == 0ull || os > best || (os == best && comp_token(oc) < comp_token(bestc)))) {
      best = os;
      bestc = oc;
    }
  }
  const float margin = 1e-4f + 2e-6f * fabsf(best);
  const float floor_s = best - margin;
  int close = 0;
  for (int r = tid; r < kept; r += SB) close += sm.s32[r] >= floor_s ? 1 : 0;
  close = __reduce_add_sync(FULL_MASK, close);
  if (tid == 0) sm.cnt = 0;
  __syncthreads();
  if (lane == 0 && close) atomicAdd(&sm.cnt, (uint32_t)close);
  __syncthreads();
  const bool screened = isfinite(best) && sm.cnt == 1u;
  __syncthreads();
  if (screened) return bestc;
  // fp64 scores of the contenders (every kept rank when the screen cannot
  // decide at all)
  const bool all = !isfinite(best);
  double ds = 0.0;
  int did = -1;
  for (int r = tid; r < kept; r += SB) {
    if (all || sm.s32[r] >= floor_s) {
      const uint64_t cc = sm.sortbuf[r];
      const int tok = comp_token(cc);
      const double s = comp_x(cc, P.temperature) + gumbel(P, tok);
      if (better(s, tok, ds, did)) {
        ds = s;
        did = tok;
      }
    }
  }
  const int id = block_argmax(ds, did, sm);
  // its composite: the kept rank holding that token
  for (int r = tid; r < kept; r += SB)
    if (comp_token(sm.sortbuf[r]) == id) sm.red_u64[0] = sm.sortbuf[r];
  __syncthreads();
  const uint64_t c = sm.red_u64[0];
  __syncthreads();
  return c;
}

// With log-probs requested (and not greedy), leaves the kept mass relative
// to the row maximum, that maximum's x and the sampled token's x in
// sm.s_kept, sm.m_row and sm.xbest.
__device__ int finish_row(const RowView &rv, int V, int nch, const RowParams &P,
                          const ChunkRec *recs, SampSmem &sm) {
  const int tid = threadIdx.x;
  if (P.mode == MODE_GREEDY) {
    uint64_t best = 0;
    for (int c = 0; c < nch; ++c) best = recs[c].top1 > best ? recs[c].top1 : best;
    return comp_token(best);
  }
  uint64_t top1 = 0;
  for (int c = 0; c < nch; ++c) top1 = recs[c].top1 > top1 ? recs[c].top1 : top1;
  if (P.mode == MODE_ALL) {
    double bs = 0.0;
    int bid = -1;
    uint32_t bkey = 0;
    for (int c = 0; c < nch; ++c)
      if (better(recs[c].gscore, recs[c].gid, bs, bid)) {
        bs = recs[c].gscore;
        bid = recs[c].gid;
        bkey = recs[c].gkey;
      }
    if (P.lp_proc) {
      // the kept mass is the whole row's: the chunks' normalisers
      const Exp2Ctx ctx = exp2_ctx(P.c2h, P.c2l, key_value((uint32_t)(top1 >> 32)));
      const DF z = row_normaliser(recs, nch, ctx, sm);
      if (tid == 0) {
        sm.s_kept = (double)z.h + (double)z.l;
        sm.m_row = comp_x(top1, P.temperature);
        sm.xbest = (double)key_value(bkey) / (double)P.temperature;
      }
      __syncthreads();
    }
    return bid;
  }
  if (P.mode == MODE_GENERAL) return general_sample(rv, V, P, top1, -1.0, sm);

  // candidate modes: the sorted prefix of the union of the chunks'
  // candidates, extended only as far as the decision reads
  const int nc = P.nc;
  const int nu = nch * nc;
  const bool full = P.mode == MODE_TOPP_FULL;
  const bool topp = P.top_p < 1.0f;
  const bool minp = P.min_p > 0.0f;
  if (tid == 0) sm.cnt = 0;
  __syncthreads();
  if (tid < nch) atomicAdd(&sm.cnt, (uint32_t)recs[tid].ncand);
  __syncthreads();
  const int nreal = (int)sm.cnt;
  // ranks the decision may read: the top-k, or for top-p over the whole
  // vocabulary up to NCAND candidates (past them: the general path)
  const int nv = min(full ? NCAND : P.K, nreal);
  __syncthreads();
  const Exp2Ctx ctx = exp2_ctx(P.c2h, P.c2l, key_value((uint32_t)(top1 >> 32)));
  // top-p over the whole vocabulary without min_p: Z is the whole row's
  DF Z = {0.0f, 0.0f};
  const bool z_row = full && !minp;
  if (z_row) Z = row_normaliser(recs, nch, ctx, sm);

  int M = full ? min(64, nv) : nv;
  int have = 0;  // ranks whose e and noise are in shared memory
  int kept = 0, kp = nv;
  bool general = false;
  for (;;) {
    // the sorted prefix [0, M)
    const bool fast = nu <= UNION_MAX && M <= SB && union_top_n(recs, nc, nu, M, sm);
    if (!fast) {
      union_sorted_slow(recs, nc, nu, nv, sm);
      M = nv;
    }
    // e_r = 2^(t_r - t_0) and the fp32 noise of the new ranks
    for (int r = have + tid; r < M; r += SB) {
      const uint64_t cc = sm.sortbuf[r];
      const DF e = df_exp2_rel(key_value((uint32_t)(cc >> 32)), ctx, sm.e2h, sm.e2l);
      sm.eh[r] = e.h;
      sm.el[r] = e.l;
      sm.g32[r] = gumbel32(P, comp_token(cc));
    }
    have = M;
    __syncthreads();
    // decision over [0, M) by warp 0: 0 = decided, 1 = extend, 2 = general
    if (tid < 32) {
      int state = 0, k_p = M, k_t = M;
      if (minp) {
        const int b = minp_boundary_warp(sm, 0, M, P.min_p);
        if (b >= 0) {
          k_p = b;
        } else if (M < nv) {
          state = 1;
        } else {
          k_p = nv;
          if (full && nv < V) state = 2;  // the boundary lies beyond the candidates
        }
      } else if (!full) {
        k_p = nv;  // the top-k
      }
      if (state == 0 && topp) {
        DF z = Z;
        if (!z_row) {
          // the normaliser over the ranks that pass top-k and min_p (one warp,
          // a fixed order: lanes in rank order, then a xor tree)
          DF part = {0.0f, 0.0f};
          for (int r = tid; r < k_p; r += 32) part = df_add(part, DF{sm.eh[r], sm.el[r]});
#pragma unroll
          for (int off = 16; off; off >>= 1) part = df_add(part, df_shfl_xor(part, off));
          z = part;
        }
        k_t = topp_cut_warp(sm, k_p, df_mul_f(z, P.top_p));
        if (k_t == k_p && !minp && full) {
          // no cut within the candidates read so far
          if (M < nv) state = 1;
          else if (nv < V) state = 2;
        }
        if (tid == 0) {
          sm.zh = z.h;
          sm.zl = z.l;
        }
      } else {
        k_t = k_p;
      }
      if (tid == 0) {
        sm.flag = state;
        sm.kp = k_p;
        sm.kept = k_t;
      }
    }
    __syncthreads();
    const int state = sm.flag;
    kp = sm.kp;
    kept = sm.kept;
    Z = DF{sm.zh, sm.zl};
    __syncthreads();
    if (state == 2) {
      general = true;
      break;
    }
    if (state == 0) break;
    M = min(2 * M, nv);
  }
  // The extracted prefix is the exact global order over the prefix the
  // decision read (the kept set; the ranks through the min_p boundary; for
  // top-k the K survivors) unless a chunk that holds more tokens than it
  // gave has its bound strictly inside that prefix.  The top-k also needs K
  // candidates in the union.
  if (!general) {
    const int decided = !full ? nv : (minp ? min(kp + 1, nv) : kept);
    const uint64_t last = sm.sortbuf[decided - 1];
    __syncthreads();
    if (tid == 0) sm.flag = (!full && P.K > nreal) ? 1 : 0;
    __syncthreads();
    if (tid < nch && recs[tid].thr > last) sm.flag = 1;
    __syncthreads();
    general = sm.flag != 0;
    __syncthreads();
  }
  if (general) {
    const double zk = z_row ? (double)Z.h + (double)Z.l : -1.0;
    return general_sample(rv, V, P, top1, zk, sm);
  }
  const uint64_t win = gumbel_argmax_sorted(P, kept, sm);
  if (P.lp_proc) {
    DF part = {0.0f, 0.0f};
    for (int r = tid; r < kept; r += SB) part = df_add(part, DF{sm.eh[r], sm.el[r]});
    const DF sk = block_sum_df(part, sm);
    if (tid == 0) {
      sm.s_kept = (double)sk.h + (double)sk.l;
      sm.m_row = comp_x(sm.sortbuf[0], P.temperature);
      sm.xbest = comp_x(win, P.temperature);
    }
    __syncthreads();
  }
  return comp_token(win);
}

// ---------------------------------------------------------------------------
// row parameters
// ---------------------------------------------------------------------------
// min_p > 0 turns on the min_p filter; lp_proc asks for the processed
// log-prob (the penalty window and the raw log-prob are set by the caller)
__device__ __forceinline__ RowParams row_params(int V, uint64_t seed, int64_t step, float temp,
                                                int32_t top_k, float top_p, uint32_t salt,
                                                float min_p = 0.0f, int lp_proc = 0) {
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
  else if (P.K <= NCAND)
    P.mode = MODE_TOPK_SMALL;
  else if (P.K == V)
    P.mode = (top_p < 1.0f || min_p > 0.0f) ? MODE_TOPP_FULL : MODE_ALL;
  else
    P.mode = MODE_GENERAL;
  P.min_p = min_p;
  P.pen = 1.0f;
  P.n_pen = 0;
  P.hist = nullptr;
  P.hist_len = 0;
  P.hist_cap = 1;
  P.lp_raw = 0;
  P.lp_proc = P.mode == MODE_GREEDY ? 0 : lp_proc;
  // the whole row's normaliser: top-p over it, or the kept mass of "keep
  // everything"; min_p takes its normaliser from the candidates instead
  P.need_z = (P.mode == MODE_TOPP_FULL && !(min_p > 0.0f)) || (P.mode == MODE_ALL && P.lp_proc);
  // candidates per chunk: enough that the union can hold the top-k (or the
  // 512 tokens top-p over the whole vocabulary may read), and at least 64
  const int kcap = P.mode == MODE_TOPK_SMALL ? P.K : NCAND;
  const int nch = (V + CHUNK - 1) / CHUNK;
  P.nc = min(kcap, max(NC_MIN, (kcap + nch - 1) / nch));
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
  // further controls (null: off)
  const float *min_p;          // [num_slots]
  const float *rep_penalty;    // [num_slots]
  const int32_t *rep_window;   // [num_slots] (null: the whole history)
  int32_t *history;            // [num_slots][hist_cap] ring of sampled tokens
  int32_t *hist_len;           // [num_slots]
  int hist_cap;
  float *lp_raw;               // [B]
  float *lp_proc;              // [B]
  uint32_t *pbits;             // [B][nch * CHUNK / 32] penalty bitmaps
};

__device__ __forceinline__ RowParams sample_row_params(const SampleArgs &a, int slot) {
  RowParams P = row_params(a.vocab, a.seeds[slot], a.steps[slot], a.temperature[slot],
                           a.top_k[slot], a.top_p[slot], a.salt,
                           a.min_p != nullptr ? a.min_p[slot] : 0.0f, a.lp_proc != nullptr);
  P.lp_raw = a.lp_raw != nullptr;
  const float pen = a.rep_penalty != nullptr ? a.rep_penalty[slot] : 1.0f;
  if (a.history != nullptr && pen != 1.0f) {
    // the window: the last min(window, length, capacity) tokens
    const int64_t len = a.hist_len[slot];
    const int32_t w = a.rep_window != nullptr ? a.rep_window[slot] : -1;
    int64_t n = len < a.hist_cap ? len : (int64_t)a.hist_cap;
    if (w >= 0 && w < n) n = w;
    if (n > 0) {
      P.n_pen = (int)n;
      P.pen = pen;
      P.hist = a.history + (int64_t)slot * a.hist_cap;
      P.hist_len = len;
      P.hist_cap = a.hist_cap;
    }
  }
  return P;
}

__device__ __forceinline__ uint32_t *row_pbits(const SampleArgs &a, int b) {
  return a.pbits != nullptr ? a.pbits + (int64_t)b * a.nch * (CHUNK / 32) : nullptr;
}

__global__ void __launch_bounds__(SB) sample_chunk_kernel(const SampleArgs a) {
  __shared__ SampSmem sm;
  const int b = blockIdx.y;
  const int c = blockIdx.x;
  // launched behind its predecessor on the stream (programmatic dependent
  // launch): nothing is read before that grid has completed
  pdl_wait();
  // the logits first (every row of the batch is readable), so that their
  // loads overlap the row's flags and settings
  float raw[EPT];
  load_chunk(a.logits + (int64_t)b * a.row_stride, a.vocab, c, raw);
  if (!a.active[b]) return;
  const int slot = a.slots[b];
  if (slot < 0 || slot >= a.num_slots) return;
  load_exp2_table(sm);  // read after the first barrier of the chunk pass
  const RowParams P = sample_row_params(a, slot);
  chunk_pass(raw, a.logits + (int64_t)b * a.row_stride, a.vocab, c, P,
             a.recs + (int64_t)b * a.nch + c, row_pbits(a, b), sm, a.err);
  // the finish kernel may be scheduled once every chunk CTA is here (late,
  // so that its waiting CTAs do not take SM room from the chunk pass)
  pdl_trigger();
}

__device__ __forceinline__ void sample_skip_row(const SampleArgs &a, int b) {
  a.out_tok[b] = 0;
  a.out_kind[b] = PKV_KIND_OTHER;
  if (a.lp_raw != nullptr) a.lp_raw[b] = 0.0f;
  if (a.lp_proc != nullptr) a.lp_proc[b] = 0.0f;
}

__global__ void __launch_bounds__(SB) sample_finish_kernel(const SampleArgs a) {
  __shared__ SampSmem sm;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  pdl_wait();  // the chunk records (and everything before them)
  if (!a.active[b]) {
    if (tid == 0) sample_skip_row(a, b);
    return;
  }
  const int slot = a.slots[b];
  if (slot < 0 || slot >= a.num_slots) {
    if (tid == 0) {
      sample_skip_row(a, b);
      report(a.err, PKV_DEV_ERR_SLOT);
    }
    return;
  }
  load_exp2_table(sm);  // read after finish_row's first barrier
  const RowParams P = sample_row_params(a, slot);
  const float *row = a.logits + (int64_t)b * a.row_stride;
  const ChunkRec *recs = a.recs + (int64_t)b * a.nch;
  const RowView rv = {row, P.n_pen > 0 ? row_pbits(a, b) : nullptr, P.pen};
  const int tok = finish_row(rv, a.vocab, a.nch, P, recs, sm);
  double lse_raw = 0.0;
  if (P.lp_raw) {
    // log-sum-exp of the unprocessed row: the chunks' partials rescaled to
    // the row maximum in parallel, added in chunk order
    float rm = recs[0].rmax;
    for (int c = 1; c < a.nch; ++c) rm = fmaxf(rm, recs[c].rmax);
    __syncthreads();
    if (tid < a.nch)
      sm.red_d[tid] = ((double)recs[tid].rzh + (double)recs[tid].rzl) *
                      exp((double)recs[tid].rmax - (double)rm);
    __syncthreads();
    if (tid == 0) {
      double z = 0.0;
      for (int c = 0; c < a.nch; ++c) z += sm.red_d[c];
      lse_raw = (double)rm + log(z);
    }
  }
  if (tid == 0) {
    a.out_tok[b] = tok;
    a.out_kind[b] = kind_of(tok, a.stop_tokens, a.n_stop, a.audio_lo, a.audio_hi);
    if (a.lp_raw != nullptr) a.lp_raw[b] = (float)((double)row[tok] - lse_raw);
    if (a.lp_proc != nullptr)
      a.lp_proc[b] = P.mode == MODE_GREEDY ? 0.0f : (float)((sm.xbest - sm.m_row) - log(sm.s_kept));
    if (a.advance) {
      a.steps[slot] = P.step + 1;
      if (a.history != nullptr) {
        const int32_t len = a.hist_len[slot];
        if (len < 0) {
          report(a.err, PKV_DEV_ERR_HISTORY);
        } else {
          a.history[(int64_t)slot * a.hist_cap + len % a.hist_cap] = tok;
          a.hist_len[slot] = len + 1;
        }
      }
    }
  }
}

struct FrameArgs {
  const float *ctrl;  // [B][ctrl_vocab] control logits, or null (no channel 0)
  int ctrl_vocab;
  int ctrl_nch;
  int32_t stop_ctrl;
  int row_w;          // ints per output row: n_cb, or 1 + n_cb with a control channel
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
  int32_t *out = a.out_codes + (int64_t)b * a.row_w;
  pdl_wait();  // the predecessor's writes (the sampler's step counters)
  if (!a.active[b]) {
    for (int j = tid; j < a.row_w; j += SB) out[j] = 0;
    if (tid == 0) a.out_kind[b] = PKV_KIND_OTHER;
    return;
  }
  const int slot = a.slots[b];
  if (slot < 0 || slot >= a.num_slots) {
    for (int j = tid; j < a.row_w; j += SB) out[j] = 0;
    if (tid == 0) {
      a.out_kind[b] = PKV_KIND_OTHER;
      report(a.err, PKV_DEV_ERR_SLOT);
    }
    return;
  }
  load_exp2_table(sm);  // read after the first barrier of the chunk pass
  const int64_t step = a.steps[slot];
  ChunkRec *recs = a.recs + (int64_t)b * (a.nch > a.ctrl_nch ? a.nch : a.ctrl_nch);
  if (a.ctrl != nullptr) {
    // channel 0: the stop/continue sample (salt 0); a stop ends the frame
    const float *crow = a.ctrl + (int64_t)b * a.ctrl_vocab;
    const RowParams P = row_params(a.ctrl_vocab, a.seeds[slot], step, a.temperature[slot],
                                   a.top_k[slot], a.top_p[slot], 0u);
    for (int c = 0; c < a.ctrl_nch; ++c) {
      float raw[EPT];
      load_chunk(crow, a.ctrl_vocab, c, raw);
      chunk_pass(raw, crow, a.ctrl_vocab, c, P, recs + c, nullptr, sm, a.err);
      __syncthreads();
    }
    const int tok = finish_row(RowView{crow, nullptr, 1.0f}, a.ctrl_vocab, a.ctrl_nch, P, recs, sm);
    if (tid == 0) {
      out[0] = tok;
      sm.token = tok;
    }
    __syncthreads();
    const bool stop = sm.token == a.stop_ctrl;
    __syncthreads();
    if (stop) {
      for (int j = 1 + tid; j < a.row_w; j += SB) out[j] = PKV_CODE_PAD;
      if (tid == 0) {
        a.out_kind[b] = PKV_KIND_STOP;
        a.steps[slot] = step + 1;
      }
      return;
    }
  }
  int32_t *codes = out + (a.row_w - a.n_cb);
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
    for (int c = 0; c < a.nch; ++c) {
      float raw[EPT];
      load_chunk(row, V, c, raw);
      chunk_pass(raw, row, V, c, P, recs + c, nullptr, sm, a.err);
      __syncthreads();
    }
    const int tok = finish_row(RowView{row, nullptr, 1.0f}, V, a.nch, P, recs, sm);
    if (tid == 0) {
      codes[j] = tok;
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

// the chunk records, then one penalty bitmap of nch * CHUNK bits per row
extern "C" size_t pkv_sample_ext_workspace_bytes(int batch, int vocab) {
  using namespace pkv;
  if (batch <= 0 || vocab <= 0) return 0;
  return pkv_sample_workspace_bytes(batch, vocab) +
         align_up((size_t)batch * chunks_for(vocab) * (CHUNK / 8), 256);
}

static size_t frame_ws_bytes(int batch, int vocab, int ctrl_vocab) {
  using namespace pkv;
  const int nch = chunks_for(vocab > ctrl_vocab ? vocab : ctrl_vocab);
  return align_up((size_t)batch * nch * sizeof(ChunkRec), 256) +
         align_up((size_t)batch * vocab * sizeof(float), 256);
}

extern "C" size_t pkv_frame_workspace_bytes(int n_codebooks, int batch, int vocab) {
  if (n_codebooks <= 0 || batch <= 0 || vocab <= 0) return 0;
  return frame_ws_bytes(batch, vocab, 0);
}

extern "C" size_t pkv_frame_sample_workspace_bytes(int n_codebooks, int batch, int vocab,
                                                   int ctrl_vocab) {
  if (n_codebooks <= 0 || batch <= 0 || vocab <= 0 || ctrl_vocab <= 0) return 0;
  return frame_ws_bytes(batch, vocab, ctrl_vocab);
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

static bool aligned4(const void *p) { return ((uintptr_t)p & 3u) == 0; }

static int launch_sample(const float *logits, int64_t row_stride, int batch, int vocab,
                         const int32_t *slots, const int32_t *active, int num_slots,
                         const uint64_t *seeds, int64_t *steps, const float *temperature,
                         const int32_t *top_k, const float *top_p, uint32_t salt, int advance,
                         const int32_t *stop_tokens, int n_stop, int32_t audio_lo,
                         int32_t audio_hi, int32_t *out_tok, int32_t *out_kind,
                         const pkv_sample_ext_t *ext, void *workspace, size_t workspace_bytes,
                         int32_t *err_word, void *stream) {
  using namespace pkv;
  int st = check_sampler_common(batch, vocab, slots, active, num_slots, seeds, steps, temperature,
                                top_k, top_p);
  if (st != PKV_OK) return st;
  if (!logits || !out_tok || !out_kind || row_stride < vocab) return PKV_ERR_INVALID_ARG;
  if (n_stop < 0 || (n_stop > 0 && !stop_tokens)) return PKV_ERR_INVALID_ARG;
  if (!aligned4(logits)) return PKV_ERR_INVALID_ARG;
  pkv_sample_ext_t e = {};
  if (ext != nullptr) e = *ext;
  if (e.history != nullptr && (e.hist_len == nullptr || e.hist_cap <= 0))
    return PKV_ERR_INVALID_ARG;
  if (!aligned4(e.min_p) || !aligned4(e.rep_penalty) || !aligned4(e.rep_window) ||
      !aligned4(e.history) || !aligned4(e.hist_len) || !aligned4(e.logprob_raw) ||
      !aligned4(e.logprob_proc))
    return PKV_ERR_INVALID_ARG;
  const bool penal = e.history != nullptr && e.rep_penalty != nullptr;
  const size_t need = penal ? pkv_sample_ext_workspace_bytes(batch, vocab)
                            : pkv_sample_workspace_bytes(batch, vocab);
  if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return PKV_ERR_INVALID_ARG;
  SampleArgs a{};
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
  a.min_p = e.min_p;
  a.rep_penalty = penal ? e.rep_penalty : nullptr;
  a.rep_window = e.rep_window;
  a.history = e.history;
  a.hist_len = e.history != nullptr ? e.hist_len : nullptr;
  a.hist_cap = e.history != nullptr ? e.hist_cap : 1;
  a.lp_raw = e.logprob_raw;
  a.lp_proc = e.logprob_proc;
  a.pbits = penal ? reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(workspace) +
                                                 pkv_sample_workspace_bytes(batch, vocab))
                  : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_pdl(sample_chunk_kernel, dim3((unsigned)a.nch, (unsigned)batch), dim3(SB), 0, s, a) !=
      cudaSuccess)
    return PKV_ERR_CUDA;
  if (launch_pdl(sample_finish_kernel, dim3((unsigned)batch), dim3(SB), 0, s, a) != cudaSuccess)
    return PKV_ERR_CUDA;
  return launch_status();
}

extern "C" int pkv_seeded_sample(const float *logits, int64_t row_stride, int batch, int vocab,
                                 const int32_t *slots, const int32_t *active, int num_slots,
                                 const uint64_t *seeds, int64_t *steps, const float *temperature,
                                 const int32_t *top_k, const float *top_p, uint32_t salt,
                                 int advance, const int32_t *stop_tokens, int n_stop,
                                 int32_t audio_lo, int32_t audio_hi, int32_t *out_tok,
                                 int32_t *out_kind, void *workspace, size_t workspace_bytes,
                                 int32_t *err_word, void *stream) {
  return launch_sample(logits, row_stride, batch, vocab, slots, active, num_slots, seeds, steps,
                       temperature, top_k, top_p, salt, advance, stop_tokens, n_stop, audio_lo,
                       audio_hi, out_tok, out_kind, nullptr, workspace, workspace_bytes, err_word,
                       stream);
}

extern "C" int pkv_seeded_sample_ext(const float *logits, int64_t row_stride, int batch,
                                     int vocab, const int32_t *slots, const int32_t *active,
                                     int num_slots, const uint64_t *seeds, int64_t *steps,
                                     const float *temperature, const int32_t *top_k,
                                     const float *top_p, uint32_t salt, int advance,
                                     const int32_t *stop_tokens, int n_stop, int32_t audio_lo,
                                     int32_t audio_hi, int32_t *out_tok, int32_t *out_kind,
                                     const pkv_sample_ext_t *ext, void *workspace,
                                     size_t workspace_bytes, int32_t *err_word, void *stream) {
  return launch_sample(logits, row_stride, batch, vocab, slots, active, num_slots, seeds, steps,
                       temperature, top_k, top_p, salt, advance, stop_tokens, n_stop, audio_lo,
                       audio_hi, out_tok, out_kind, ext, workspace, workspace_bytes, err_word,
                       stream);
}

static int launch_frame(const float *ctrl, int ctrl_vocab, int32_t stop_ctrl, const float *base,
                        const float *fb, int n_codebooks, int batch, int vocab,
                        const int32_t *slots, const int32_t *active, int num_slots,
                        const uint64_t *seeds, int64_t *steps, const float *temperature,
                        const int32_t *top_k, const float *top_p, int32_t *out, int32_t *out_kind,
                        void *workspace, size_t workspace_bytes, int32_t *err_word, void *stream) {
  using namespace pkv;
  int st = check_sampler_common(batch, vocab, slots, active, num_slots, seeds, steps, temperature,
                                top_k, top_p);
  if (st != PKV_OK) return st;
  if (!base || !out || !out_kind || n_codebooks <= 0) return PKV_ERR_INVALID_ARG;
  if (((uintptr_t)base & 3u) != 0 || ((uintptr_t)fb & 3u) != 0 || ((uintptr_t)ctrl & 3u) != 0)
    return PKV_ERR_INVALID_ARG;
  if (ctrl_vocab > MAX_CHUNKS * CHUNK) return PKV_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < frame_ws_bytes(batch, vocab, ctrl ? ctrl_vocab : 0))
    return PKV_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return PKV_ERR_INVALID_ARG;
  FrameArgs a;
  a.ctrl = ctrl;
  a.ctrl_vocab = ctrl ? ctrl_vocab : 0;
  a.ctrl_nch = ctrl ? chunks_for(ctrl_vocab) : 0;
  a.stop_ctrl = stop_ctrl;
  a.row_w = (ctrl ? 1 : 0) + n_codebooks;
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
  a.out_codes = out;
  a.out_kind = out_kind;
  a.recs = static_cast<ChunkRec *>(workspace);
  const int rec_nch = a.nch > a.ctrl_nch ? a.nch : a.ctrl_nch;
  a.rows = reinterpret_cast<float *>(static_cast<unsigned char *>(workspace) +
                                     align_up((size_t)batch * rec_nch * sizeof(ChunkRec), 256));
  a.err = err_word;
  if (launch_pdl(frame_kernel, dim3((unsigned)batch), dim3(SB), 0,
                 static_cast<cudaStream_t>(stream), a) != cudaSuccess)
    return PKV_ERR_CUDA;
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
  return launch_frame(nullptr, 0, 0, base, fb, n_codebooks, batch, vocab, slots, active, num_slots,
                      seeds, steps, temperature, top_k, top_p, out_codes, out_kind, workspace,
                      workspace_bytes, err_word, stream);
}

extern "C" int pkv_frame_sample(const float *ctrl_logits, int ctrl_vocab, int32_t stop_ctrl,
                                const float *base, const float *fb, int n_codebooks, int batch,
                                int vocab, const int32_t *slots, const int32_t *active,
                                int num_slots, const uint64_t *seeds, int64_t *steps,
                                const float *temperature, const int32_t *top_k,
                                const float *top_p, int32_t *out_rows, int32_t *out_kind,
                                void *workspace, size_t workspace_bytes, int32_t *err_word,
                                void *stream) {
  if (!ctrl_logits || ctrl_vocab <= 0 || stop_ctrl < 0 || stop_ctrl >= ctrl_vocab)
    return PKV_ERR_INVALID_ARG;
  return launch_frame(ctrl_logits, ctrl_vocab, stop_ctrl, base, fb, n_codebooks, batch, vocab,
                      slots, active, num_slots, seeds, steps, temperature, top_k, top_p, out_rows,
                      out_kind, workspace, workspace_bytes, err_word, stream);
}
