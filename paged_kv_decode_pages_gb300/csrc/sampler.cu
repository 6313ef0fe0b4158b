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
// its own logits and slot state only.  The order is exact (integer keys of
// the fp32 logits); the top-p and min_p cuts are taken on double-float
// sums whose terms are within 3e-9 of themselves, so they can differ from
// the fp64 definition only at near-ties; the Gumbel argmax is screened in
// fp32 and decided in fp64 among the ranks within the screen's error margin
// (see "Arithmetic of the decision" below).
//
// Structure:
//  * order key: the fp32 logit mapped to a uint32 that sorts like the float
//    (-0 folded onto +0); composite = key << 32 | ~token, so a larger
//    composite comes first in (value desc, id asc) order, and composites
//    are unique.
//  * chunk pass (one CTA per 8192-token chunk of a row; the chunk is staged
//    in shared memory -- bulk copies from one thread on an mbarrier when it
//    is 16-byte aligned, else cp.async from every thread -- and turned into
//    order keys in place): the chunk's nc largest composites, nc =
//    min(kcap, max(16, ceil(kcap / chunks))) with kcap = the top-k, or 512
//    for top-p over the whole vocabulary, and the smallest of them.  For
//    nc <= 256 they come from a lower bound taken from the warps' largest
//    thread maxima (select_bound: a top-2 / top-4 reduction over the lanes,
//    or a sort over the lanes), a per-warp gather of the keys at or above
//    it and exact rank counting over those, in descending order; otherwise,
//    or when a warp gathers more than 128, from a radix select over 8-bit
//    digits.  For top-p over the whole vocabulary, the partial normaliser
//    sum exp(x - x_chunkmax) = sum 2^(logit * log2(e) / T - t_chunkmax) in
//    double-float arithmetic (fp32 pairs, two terms at a time on packed
//    f32x2 operations): Tang's table-driven exp2 (ACM TOMS 15(2), 1989)
//    with a double-float table of 2^(j/32) and a degree-4 polynomial, each
//    term within 3e-9 of itself, summed with exact two-sum corrections --
//    on this GPU one fp64 warp instruction costs as much issue time as
//    several dozen fp32 ones, and this is the only per-logit transcendental
//    of the path; for "keep everything", the chunk's Gumbel argmax.  When
//    two CTAs per chunk fit on the SMs at once, a second CTA per chunk
//    computes the normaliser partials (the same arithmetic) while the first
//    selects.  The chunking depends on the vocabulary only.
//  * finish (one CTA per row, released as soon as the last chunk CTA has
//    started): the chunks' candidates in order -- the whole union sorted by
//    a register / shuffle bitonic merge of the sorted lists when it fits
//    1024 entries, else a pairwise merge of the lists' heads, or a radix
//    select and a sort from the records; min_p, then top-p with
//    double-float prefix sums in sorted order (a top-k of at most 64 decided
//    by one warp); the Gumbel argmax (arithmetic below).  The
//    sorted candidates are the exact global order over the prefix the
//    decision read unless a chunk holding more tokens than it gave has its
//    smallest candidate strictly inside that prefix; such rows, and rows
//    whose kept set is not decided by kcap tokens (top-k > 512, or top-p
//    needing more than 512 tokens), take an exact general path that streams
//    the row: radix select of the top-k threshold and progressive sorted
//    extraction until the top-p crossing.
//  * a vocabulary of one chunk runs the chunk pass and the finish in one
//    CTA per row (sample_single_kernel), with the same arithmetic.
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
#include <stddef.h>

#include <atomic>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int SB = 256;                 // threads per sampler CTA
constexpr int CHUNK = 8192;             // tokens per chunk
constexpr int NCAND = 512;              // most candidates kept per chunk
constexpr int NC_MIN = 16;              // least candidates kept per chunk
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
  int32_t sorted;      // cand[0, ncand) is in descending order
  int32_t pad_;
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

// The same two computations on packed fp32 pairs, each half exactly the
// scalar function's operations (so each half's result is the scalar one):
// df_exp2_rel of two values, df_accumulate of two accumulators.
struct DF2 {
  f32x2 h, l;
};
__device__ __forceinline__ DF2 df2_exp2_rel(f32x2 v, const Exp2Ctx &c, const float *tab_h,
                                            const float *tab_l) {
  constexpr f32x2 SIGN = 0x8000000080000000ull;
  const f32x2 ph = fmul2(v, pack2(c.c2h, c.c2h));
  const f32x2 pl = ffma2(v, pack2(c.c2l, c.c2l), ffma2(v, pack2(c.c2h, c.c2h), ph ^ SIGN));
  // s = ph + (-th), exactly, as df_two_sum
  const f32x2 nth = pack2(-c.th, -c.th);
  const f32x2 sh = fadd2(ph, nth);
  const f32x2 bb = fsub2(sh, ph);
  const f32x2 sl = fadd2(fsub2(ph, fsub2(sh, bb)), fsub2(nth, bb));
  const f32x2 tlow = fsub2(fadd2(sl, pl), pack2(c.tl, c.tl));
  const f32x2 magic = pack2(12582912.0f, 12582912.0f);
  const f32x2 y = ffma2(sh, pack2(32.0f, 32.0f), magic);
  const f32x2 g = ffma2(fsub2(y, magic), pack2(-0.03125f, -0.03125f), sh);
  const f32x2 r = fadd2(g, tlow);
  const f32x2 u = ffma2(r, pack2(LN2_H, LN2_H), fmul2(r, pack2(LN2_L, LN2_L)));
  f32x2 q = ffma2(u, pack2(1.0f / 24.0f, 1.0f / 24.0f), pack2(1.0f / 6.0f, 1.0f / 6.0f));
  q = ffma2(q, u, pack2(0.5f, 0.5f));
  q = ffma2(q, u, pack2(1.0f, 1.0f));
  q = fmul2(q, u);
  // n = rint(32 s.h) = 32 k + j per half (unsigned: a half out of range
  // gives garbage here, which is masked off below)
  const float2 yy = unpack2(y);
  const uint32_t n0 = (uint32_t)__float_as_int(yy.x) - 0x4B400000u;
  const uint32_t n1 = (uint32_t)__float_as_int(yy.y) - 0x4B400000u;
  const int j0 = (int)(n0 & 31u), j1 = (int)(n1 & 31u);
  const int k0 = (int)n0 >> 5, k1 = (int)n1 >> 5;
  const f32x2 t0 = pack2(tab_h[j0], tab_h[j1]);
  const f32x2 b = ffma2(t0, q, pack2(tab_l[j0], tab_l[j1]));
  const f32x2 eh = fadd2(t0, b);
  const f32x2 el = fsub2(b, fsub2(eh, t0));
  const f32x2 sc = pack2(__int_as_float((int)(((uint32_t)(k0 + 127)) << 23)),
                         __int_as_float((int)(((uint32_t)(k1 + 127)) << 23)));
  // 0 for a half below 2^-125 or with a -inf value
  const float2 s2 = unpack2(sh);
  const f32x2 keep = (s2.x > -125.0f ? 0x00000000ffffffffull : 0ull) |
                     (s2.y > -125.0f ? 0xffffffff00000000ull : 0ull);
  return DF2{fmul2(eh, sc) & keep, fmul2(el, sc) & keep};
}
__device__ __forceinline__ void df2_accumulate(DF2 &acc, DF2 e) {
  const f32x2 sh = fadd2(acc.h, e.h);
  const f32x2 bb = fsub2(sh, acc.h);
  const f32x2 sl = fadd2(fsub2(acc.h, fsub2(sh, bb)), fsub2(e.h, bb));
  acc.h = sh;
  acc.l = fadd2(acc.l, fadd2(sl, e.l));
}


// ---------------------------------------------------------------------------
// Philox4x64-10 and Gumbel noise
// ---------------------------------------------------------------------------
// (rolled, out of line: the sampler's kernels run most of their code once
// per call, so code size rather than issue count sets their latency)
__device__ __noinline__ uint64_t philox_word0(uint64_t seed, uint32_t salt, uint64_t token,
                                              uint64_t step) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
  uint64_t c0 = token, c1 = step, c2 = 0, c3 = 0;
  uint64_t k0 = seed, k1 = salt;
#pragma unroll 1
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

__device__ __noinline__ double gumbel(const RowParams &P, int token) {
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

// order_key without the checks: the fp32 bits mapped to a uint32 that
// sorts like the float, -0 folded onto +0.  A NaN maps outside
// [key(-inf), key(+inf)]; keys_fix_bad() repairs those.
__device__ __forceinline__ uint32_t fast_key(uint32_t u) {
  const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
  return k == 0x7fffffffu ? 0x80000000u : k;
}
constexpr uint32_t KEY_NEG_INF = 0x007fffffu, KEY_POS_INF = 0xff800000u;

__device__ __forceinline__ float key_value(uint32_t key) {
  const uint32_t u = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
  return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t composite(uint32_t key, int token) {
  return ((uint64_t)key << 32) | (uint32_t)(~(uint32_t)token);
}
__device__ __forceinline__ int comp_token(uint64_t c) { return (int)(~(uint32_t)c); }
__device__ __noinline__ double comp_x(uint64_t c, float temperature) {
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
constexpr int UNION_MAX = 2048;  // largest candidate union a finish stages in shared memory

struct ChunkScratch {
  uint32_t keys[CHUNK];          // the chunk: fp32 logits, then their order keys
  uint32_t penbits[CHUNK / 32];  // penalised tokens of the chunk
};
struct DecideScratch {
  float eh[NCAND], el[NCAND];    // 2^(t_r - t_0) of the sorted candidates, double-float
  float g32[NCAND];              // their fp32 Gumbel noise
  float s32[NCAND];              // their fp32 scores
};
struct FinishScratch {
  uint64_t uni[UNION_MAX];       // the chunks' candidates, packed in chunk order
  union {
    uint64_t gather[GEN_BLOCK];  // candidates above a selection bound
    DecideScratch d;             // (after the selection)
    double es[GEN_BLOCK];        // general path
  } a;
  uint64_t mrg[GEN_BLOCK];       // the other buffer of the pairwise merges
};

// A chunk of at most SREC_MAX_V keys leaves the merge buffer of the shared
// union free, room for one chunk record.
constexpr int SREC_MAX_V = (int)(sizeof(FinishScratch) - GEN_BLOCK * sizeof(uint64_t)) / 4;
static_assert(sizeof(ChunkRec) <= GEN_BLOCK * sizeof(uint64_t), "a chunk record fits the merge buffer");
static_assert(offsetof(FinishScratch, mrg) == sizeof(FinishScratch) - GEN_BLOCK * sizeof(uint64_t),
              "the merge buffer ends the finish scratch");

struct __align__(16) SampSmem {
  float e2h[32], e2l[32];  // the 2^(j/32) table
  float wh[SB / 32], wl[SB / 32];
  uint32_t hist[256];
  uint64_t red_u64[SB / 32];
  uint64_t red_u64b[SB / 32];
  uint32_t offer[SB / 32], wtop[SB / 32];
  double wd[SB / 32];                        // per-warp fp64 partials
  int32_t wi[SB / 32];                       // per-warp ids
  int32_t cn[MAX_CHUNKS], coff[MAX_CHUNKS];  // candidates per chunk and their offsets
  int32_t csorted[MAX_CHUNKS];               // whether each chunk's list is in order
  int32_t wcnt[SB / 32];                     // per-warp list lengths
  uint64_t htop[MAX_CHUNKS], hthr[MAX_CHUNKS];  // the chunks' largest composites and bounds
  float fh[MAX_CHUNKS], fl[MAX_CHUNKS];      // the chunks' rescaled normalisers
  uint64_t s_top1, s_bound;                  // over the chunks: largest composite, largest bound
  int32_t s_total, s_sorted;                 // over the chunks: candidates, all lists in order
  int32_t s_pad[2];                          // keeps the buffers below 16-byte aligned
  float wbs[SB / 32];                        // per-warp best fp32 scores
  uint64_t sel_prefix;
  uint64_t nth;      // rank_out: the composite of rank n - 1
  uint64_t first;    // rank_out: the composite of rank 0
  uint32_t sel_want;
  uint32_t sel_done;
  uint32_t cnt;
  int32_t flag;
  int32_t token;
  int32_t kept;
  int32_t done;
  int32_t kp;
  float zh, zl;      // a normaliser, double-float
  double zsum;
  double s_kept;     // mass (relative to the row maximum) of the kept tokens
  double m_row;      // x of the row maximum
  double xbest;      // x of the sampled token
  uint64_t stage_bar;  // completion of the chunk's bulk copies
  uint64_t stage_pad;  // keeps the buffers below 16-byte aligned
  uint64_t sortbuf[GEN_BLOCK];  // sorted prefixes; the chunk pass's candidate buffer
  union {
    ChunkScratch ch;
    FinishScratch fi;
  } u;
};
static_assert(sizeof(SampSmem) <= 48 * 1024, "static shared memory of one sampler CTA");
static_assert(sizeof(FinishScratch) <= sizeof(ChunkScratch), "the finish's scratch fits the chunk's");
static_assert(CHUNK == 1 << 13, "a token's chunk is token >> 13");
static_assert(offsetof(SampSmem, u) % 16 == 0 && offsetof(SampSmem, sortbuf) % 16 == 0,
              "16-byte copies into the chunk buffer and the union");

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

// Sum in a fixed order: a xor tree in each warp, then the warps in order.
__device__ __noinline__ double block_sum_d(double v, SampSmem &sm) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(FULL_MASK, v, off);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.wd[threadIdx.x >> 5] = v;
  __syncthreads();
  double r = sm.wd[0];
  for (int w = 1; w < SB / 32; ++w) r += sm.wd[w];
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

__device__ __noinline__ int block_argmax(double s, int id, SampSmem &sm,
                                         double *best_score = nullptr) {
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const double s2 = __shfl_xor_sync(FULL_MASK, s, off);
    const int i2 = __shfl_xor_sync(FULL_MASK, id, off);
    if (better(s2, i2, s, id)) {
      s = s2;
      id = i2;
    }
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    sm.wd[threadIdx.x >> 5] = s;
    sm.wi[threadIdx.x >> 5] = id;
  }
  __syncthreads();
  double bs = sm.wd[0];
  int bid = sm.wi[0];
  for (int w = 1; w < SB / 32; ++w)
    if (better(sm.wd[w], sm.wi[w], bs, bid)) {
      bs = sm.wd[w];
      bid = sm.wi[w];
    }
  if (best_score) *best_score = bs;
  __syncthreads();
  return bid;
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
// candidate selection (chunk pass and finish)
// ---------------------------------------------------------------------------
// The sampler kernels run each phase once per row or chunk, so the code they
// execute is mostly fetched cold: every new line of instructions costs an L2
// round trip.  The per-element phases are therefore short rolled loops over
// data staged in shared memory (the chunk's keys, the candidate union), not
// loops unrolled over register arrays, and the rarely taken paths are kept
// out of the hot code.

// The Q largest of the warp's 32 values v (Q = 2 or 4), in descending order
// in every lane: five xor-shuffle rounds, each merging the lane's Q largest
// with its partner's (the k-th largest of two descending lists a, b is the
// largest of min(a[i], b[k - i]) over i, with a[0] = b[0] = +inf).  0 is
// below every key.
template <int Q>
__device__ __forceinline__ void warp_top(uint32_t v, uint32_t (&t)[Q]) {
  t[0] = v;
#pragma unroll
  for (int i = 1; i < Q; ++i) t[i] = 0u;
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    uint32_t o[Q], r[Q];
#pragma unroll
    for (int i = 0; i < Q; ++i) o[i] = __shfl_xor_sync(FULL_MASK, t[i], off);
#pragma unroll
    for (int k = 1; k <= Q; ++k) {
      uint32_t best = max(t[k - 1], o[k - 1]);  // the terms with i = k and i = 0
#pragma unroll
      for (int i = 1; i < k; ++i) best = max(best, min(t[i - 1], o[k - i - 1]));
      r[k - 1] = best;
    }
#pragma unroll
    for (int i = 0; i < Q; ++i) t[i] = r[i];
  }
}

// From the threads' largest keys m: a bound L such that at least n of the
// block's keys are >= L -- each warp offers the q-th largest of its 32
// maxima, q = ceil(n / 8) (for q <= 4 a top-q reduction over the lanes,
// else a bitonic sort over the lanes), and L is the smallest offer, so
// every warp holds q keys >= L -- and the block's largest key in *top.
// n <= SB.  All threads get both.
__device__ uint32_t select_bound(uint32_t m, int n, SampSmem &sm, uint32_t *top) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int q = (n + (SB / 32) - 1) / (SB / 32);
  uint32_t v, offer;
  if (q <= 2) {
    uint32_t t[2];
    warp_top<2>(m, t);
    v = t[0];
    offer = t[q - 1];
  } else if (q <= 4) {
    uint32_t t[4];
    warp_top<4>(m, t);
    v = t[0];
    offer = q == 3 ? t[2] : t[3];
  } else {
    v = m;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const uint32_t o = __shfl_xor_sync(FULL_MASK, v, j);
        const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
        v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
      }
    offer = __shfl_sync(FULL_MASK, v, q - 1);
    v = __shfl_sync(FULL_MASK, v, 0);
  }
  __syncthreads();  // earlier readers of the per-warp slots are done
  if (lane == 0) {
    sm.offer[warp] = offer;
    sm.wtop[warp] = v;  // the warp's largest (lane 0 after the descending sort)
  }
  __syncthreads();
  uint32_t L = sm.offer[0], t = sm.wtop[0];
#pragma unroll
  for (int w = 1; w < SB / 32; ++w) {
    L = sm.offer[w] < L ? sm.offer[w] : L;
    t = sm.wtop[w] > t ? sm.wtop[w] : t;
  }
  *top = t;
  return L;
}




// ---------------------------------------------------------------------------
// selection with independent work per thread
// ---------------------------------------------------------------------------
// One or a few sampler CTAs share an SM, so these loops are bound by the
// latency of dependent instructions rather than by issue: every thread gets
// several independent loads and sums per step (four keys per lane, eight
// comparisons per counting step, several lists per binary-search step),
// and hits are collected with warp ballots (no shared counters, no prefix
// chains).
constexpr int WCAP = GEN_BLOCK / (SB / 32);  // 128: longest per-warp list

// Appends, for the calling warp, composite(k, id0 + i) of every key
// k = keys[i] >= L among the warp's share of keys[0, cnt) (uint4 q = base +
// lane, base = warp * 32 + m * SB; the tail cnt % 4 goes to warp 0) to lst
// (positions from four ballots per step); returns the warp's count
// (warp-uniform; entries past WCAP are dropped, the count is not).
__device__ __forceinline__ int warp_collect_above(const uint32_t *keys, int cnt, int id0,
                                                  uint32_t L, uint64_t *lst) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const int nq = cnt >> 2;
  const uint4 *k4 = reinterpret_cast<const uint4 *>(keys);
  int nw = 0;
#pragma unroll 1
  for (int base = warp * 32; base < nq; base += SB) {  // the same trip count in every lane
    const int q = base + lane;
    const bool v = q < nq;
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (v) u = k4[q];
    const uint32_t um = max(max(u.x, u.y), max(u.z, u.w));
    if (__ballot_sync(FULL_MASK, v && um >= L) != 0u) {  // most steps have no hit at all
      const unsigned b0 = __ballot_sync(FULL_MASK, v && u.x >= L);
      const unsigned b1 = __ballot_sync(FULL_MASK, v && u.y >= L);
      const unsigned b2 = __ballot_sync(FULL_MASK, v && u.z >= L);
      const unsigned b3 = __ballot_sync(FULL_MASK, v && u.w >= L);
      const int n1 = nw + __popc(b0), n2 = n1 + __popc(b1), n3 = n2 + __popc(b2);
      const int id = id0 + 4 * q;
      int pos;
      if ((b0 >> lane) & 1u) {
        pos = nw + __popc(b0 & lt);
        if (pos < WCAP) lst[pos] = composite(u.x, id);
      }
      if ((b1 >> lane) & 1u) {
        pos = n1 + __popc(b1 & lt);
        if (pos < WCAP) lst[pos] = composite(u.y, id + 1);
      }
      if ((b2 >> lane) & 1u) {
        pos = n2 + __popc(b2 & lt);
        if (pos < WCAP) lst[pos] = composite(u.z, id + 2);
      }
      if ((b3 >> lane) & 1u) {
        pos = n3 + __popc(b3 & lt);
        if (pos < WCAP) lst[pos] = composite(u.w, id + 3);
      }
      nw = n3 + __popc(b3);
    }
  }
  if (warp == 0) {
    const int i = 4 * nq + lane;
    const bool hit = i < cnt && keys[i] >= L;
    const unsigned bm = __ballot_sync(FULL_MASK, hit);
    if (hit) {
      const int pos = nw + __popc(bm & lt);
      if (pos < WCAP) lst[pos] = composite(keys[i], id0 + i);
    }
    nw += __popc(bm);
  }
  return nw;
}

// The nc largest of the C distinct composites g[0, C) (16-byte aligned), in
// descending order, to out[0, min(nc, C)): each one's rank is the number of
// larger ones, counted eight at a time with two running counts.  Leaves
// rank 0 in sm.first and rank nc - 1 in sm.nth (which the caller clears).
__device__ __noinline__ void rank_count_out(const uint64_t *g, int C, int nc, uint64_t *out,
                                            SampSmem &sm) {
  const ulonglong2 *g2 = reinterpret_cast<const ulonglong2 *>(g);
  for (int e = threadIdx.x; e < C; e += SB) {
    const uint64_t x = g[e];
    int r0 = 0, r1 = 0, k = 0;
#pragma unroll 1
    for (; k + 8 <= C; k += 8) {
      const ulonglong2 a = g2[k >> 1], b = g2[(k >> 1) + 1], c = g2[(k >> 1) + 2],
                       d = g2[(k >> 1) + 3];
      r0 += (a.x > x) + (a.y > x) + (b.x > x) + (b.y > x);
      r1 += (c.x > x) + (c.y > x) + (d.x > x) + (d.y > x);
    }
    for (; k < C; ++k) r0 += g[k] > x ? 1 : 0;
    const int r = r0 + r1;
    if (r < nc) out[r] = x;
    if (r == 0) sm.first = x;
    if (r == nc - 1) sm.nth = x;
  }
}

// ---------------------------------------------------------------------------
// chunk pass
// ---------------------------------------------------------------------------
// The chunk [start, start + cnt) of `row` into buf as fp32 bits; every copy
// is issued before any is waited for.
__device__ __forceinline__ void stage_chunk_issue(const float *row, int start, int cnt,
                                                  uint32_t *buf) {
  const float *src = row + start;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0 && (cnt & 3) == 0) {
    for (int i = 4 * (int)threadIdx.x; i < cnt; i += 4 * SB) cp_async16(buf + i, src + i);
  } else {
    for (int i = (int)threadIdx.x; i < cnt; i += SB) cp_async4(buf + i, src + i);
  }
}
__device__ __forceinline__ void stage_chunk(const float *row, int start, int cnt, uint32_t *buf) {
  stage_chunk_issue(row, start, cnt, buf);
  cp_async_wait_all();
  __syncthreads();
}


// The chunk [start, start + cnt) of `row` into the chunk buffer in two
// steps, so that other work can run while the copies are in flight.
// stage_chunk_begin issues them: bulk copies from thread 0 (8 KB each, on
// one mbarrier) when the chunk starts on a 16-byte boundary and is a
// multiple of 16 bytes long, else cp.async from every thread; it returns
// which.  stage_chunk_end waits for them (a block barrier included): false
// when bulk copies did not land in time -- reported, and waited for once
// more so that none is still writing when the CTA leaves.
__device__ __forceinline__ bool stage_chunk_begin(const float *row, int start, int cnt,
                                                  SampSmem &sm) {
  const bool bulk = (reinterpret_cast<uintptr_t>(row + start) & 15u) == 0 && (cnt & 3) == 0;
  if (bulk) {
    if (threadIdx.x == 0) {
      mbar_init(&sm.stage_bar, 1);
      fence_barrier_init();
      const uint32_t bytes = 4u * (uint32_t)cnt;
      mbar_arrive_expect_tx(&sm.stage_bar, bytes);
      const unsigned char *src = reinterpret_cast<const unsigned char *>(row + start);
      unsigned char *dst = reinterpret_cast<unsigned char *>(sm.u.ch.keys);
      for (uint32_t off = 0; off < bytes; off += 8192u)
        bulk_copy_g2s(dst + off, src + off, min(8192u, bytes - off), &sm.stage_bar);
    }
  } else {
    stage_chunk_issue(row, start, cnt, sm.u.ch.keys);
  }
  return bulk;
}
__device__ __forceinline__ bool stage_chunk_end(bool bulk, SampSmem &sm, int32_t *err) {
  if (!bulk) cp_async_wait_all();
  __syncthreads();
  if (bulk && !__syncthreads_and(mbar_wait(&sm.stage_bar, 0))) {
    if (threadIdx.x == 0) report(err, PKV_DEV_ERR_TIMEOUT);
    (void)mbar_wait(&sm.stage_bar, 0);
    return false;
  }
  return true;
}

// The keys of NaN logits (outside [key(-inf), key(+inf)]) set to key(-inf):
// a NaN ranks like -inf; NaN and +inf are reported.  Returns the thread's
// largest key after the repair.
__device__ __noinline__ uint32_t keys_fix_bad(uint32_t *keys, int cnt, int32_t *err) {
  uint32_t m = 0;
  bool bad = false;
  for (int i = threadIdx.x; i < cnt; i += SB) {
    uint32_t k = keys[i];
    if (k > KEY_POS_INF || k < KEY_NEG_INF) {
      k = KEY_NEG_INF;
      keys[i] = k;
      bad = true;
    } else if (k == KEY_POS_INF) {
      bad = true;
    }
    m = k > m ? k : m;
  }
  if (bad) report(err, PKV_DEV_ERR_LOGITS);
  return m;
}


// The chunk's nc largest composites at or above the bound L, in descending
// order, to out[0, min(nc, C)) with C the number of keys >= L: each warp
// collects its own keys' hits into its own list in sortbuf, the lists are
// closed up into one, and every entry is placed by counting the larger
// ones.  Leaves rank 0 in sm.first and rank nc - 1 in sm.nth.  Returns C,
// or -1 (nothing written) when a warp holds more than WCAP hits.
__device__ __noinline__ int chunk_select_sorted(const uint32_t *keys, int cnt, int id0, uint32_t L,
                                                int nc, uint64_t *out, SampSmem &sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t *lst = sm.sortbuf + warp * WCAP;
  const int nw = warp_collect_above(keys, cnt, id0, L, lst);
  if (lane == 0) sm.wcnt[warp] = nw;
  if (threadIdx.x == 0) sm.nth = 0ull;
  if (__syncthreads_or(nw > WCAP)) return -1;
  int off = 0, C = 0;
#pragma unroll
  for (int w = 0; w < SB / 32; ++w) {
    const int c = sm.wcnt[w];
    off += w < warp ? c : 0;
    C += c;
  }
  uint64_t v[WCAP / 32];
#pragma unroll
  for (int e = 0; e < WCAP / 32; ++e) v[e] = e * 32 + lane < nw ? lst[e * 32 + lane] : 0ull;
  __syncthreads();
#pragma unroll
  for (int e = 0; e < WCAP / 32; ++e)
    if (e * 32 + lane < nw) sm.sortbuf[off + e * 32 + lane] = v[e];
  __syncthreads();
  rank_count_out(sm.sortbuf, C, nc, out, sm);
  __syncthreads();
  return C;
}

// Sum over the chunk of 2^(key_value(k) * c2 - t_max), every term in
// double-float (Tang's table-driven exp2, exact two-sum accumulation); all
// threads get it.  Each thread takes four keys at a time (a uint4) into four
// independent sums.  (Taking the terms below 2^-24 of the largest on the
// SFU in fp32 and listing only the larger ones for double-float was slower
// on every logit spread measured: the listing costs more than it saves.)
__device__ __noinline__ DF chunk_exp_sum_all(const uint32_t *keys, int cnt, const Exp2Ctx ctx,
                                             SampSmem &sm) {
  const int nq = cnt >> 2;
  const uint4 *k4 = reinterpret_cast<const uint4 *>(keys);
  // four accumulators a0..a3 (components x, y, z, w of each 16-byte load),
  // as the packed pairs (a0, a1) and (a2, a3)
  DF2 a01 = {0ull, 0ull}, a23 = {0ull, 0ull};
#pragma unroll 1
  for (int q = threadIdx.x; q < nq; q += SB) {
    const uint4 u = k4[q];
    df2_accumulate(a01, df2_exp2_rel(pack2(key_value(u.x), key_value(u.y)), ctx, sm.e2h, sm.e2l));
    df2_accumulate(a23, df2_exp2_rel(pack2(key_value(u.z), key_value(u.w)), ctx, sm.e2h, sm.e2l));
  }
  const float2 h01 = unpack2(a01.h), l01 = unpack2(a01.l), h23 = unpack2(a23.h),
               l23 = unpack2(a23.l);
  DF a0 = {h01.x, l01.x};
  const DF a1 = {h01.y, l01.y}, a2 = {h23.x, l23.x}, a3 = {h23.y, l23.y};
  for (int i = 4 * nq + (int)threadIdx.x; i < cnt; i += SB)
    df_accumulate(a0, df_exp2_rel(key_value(keys[i]), ctx, sm.e2h, sm.e2l));
  const DF lo = df_add(df_fast_two_sum(a0.h, a0.l), df_fast_two_sum(a1.h, a1.l));
  const DF hi = df_add(df_fast_two_sum(a2.h, a2.l), df_fast_two_sum(a3.h, a3.l));
  return block_sum_df(df_add(lo, hi), sm);
}

// Keep everything: the chunk's Gumbel argmax in fp64 (the definition);
// block result in *bs, *bid, *bkey (tid 0).
__device__ __noinline__ void chunk_gumbel_all(const uint32_t *keys, int start, int cnt,
                                              const RowParams P, SampSmem &sm, double *bs,
                                              int *bid, uint32_t *bkey) {
  double s0 = 0.0;
  int id0 = -1;
  uint32_t k0 = 0u;
  for (int i = (int)threadIdx.x; i < cnt; i += SB) {
    const int tok = start + i;
    const double s = (double)key_value(keys[i]) / (double)P.temperature + gumbel(P, tok);
    if (better(s, tok, s0, id0)) {
      s0 = s;
      id0 = tok;
      k0 = keys[i];
    }
  }
  double best;
  const int id = block_argmax(s0, id0, sm, &best);
  if (id0 == id && id >= 0) sm.token = (int32_t)k0;
  __syncthreads();
  *bs = best;
  *bid = id;
  *bkey = (uint32_t)sm.token;
}

// The chunk's nc largest composites (unsorted) and their bound by an exact
// radix select over 8-bit digits: for top-k above 256, or when the
// selection bound lets more than GEN_BLOCK keys through (many ties).
__device__ __noinline__ void chunk_radix_top(const uint32_t *keys, int start, int cnt, int nc,
                                             ChunkRec *rec, SampSmem &sm) {
  const int tid = threadIdx.x;
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
    for (int i = tid; i < cnt; i += SB) {
      const uint64_t cc = composite(keys[i], start + i);
      if ((cc & mask) == prefix) atomicAdd(&sm.hist[(cc >> shift) & 255u], 1u);
    }
    __syncthreads();
    select_bin(sm, shift);
    mask |= 255ull << shift;
    if (sm.sel_done) break;
  }
  const uint64_t thr = sm.sel_prefix;
  __syncthreads();
  if (tid == 0) sm.cnt = 0;
  __syncthreads();
  for (int i = tid; i < cnt; i += SB) {
    const uint64_t cc = composite(keys[i], start + i);
    if (cc >= thr) {
      const uint32_t pos = atomicAdd(&sm.cnt, 1u);
      if (pos < (uint32_t)nc) rec->cand[pos] = cc;
    }
  }
  __syncthreads();
  const int got = min((int)sm.cnt, nc);
  for (int i = got + tid; i < nc; i += SB) rec->cand[i] = 0ull;
  if (tid == 0) {
    rec->ncand = got;
    rec->thr = thr;
    rec->sorted = 0;
  }
}

// One chunk of a row: stage it, form the order keys (penalty applied), then
// per mode the chunk's largest composite, its nc largest composites with
// their bound, the normaliser partial or the Gumbel winner, into *rec.
// pbits: the row's penalty bitmap in global memory, written for this chunk
// when the row is penalised (may be null otherwise).  prestaged: the
// caller has already put the chunk's logits into sm.u.ch.keys.
// What a chunk CTA computes: everything, or (a row whose chunks each get
// two CTAs) the candidates and the rest, or the two normaliser partials
// (the raw log-softmax one and the processed one, each when asked for).
enum ChunkPart : int { PART_ALL = 0, PART_SELECT = 1, PART_NORM = 2 };

__device__ __noinline__ void chunk_pass(const float *row, int V, int c, const RowParams &P,
                                        ChunkRec *rec, uint32_t *pbits, SampSmem &sm,
                                        int32_t *err, bool prestaged = false,
                                        int part = PART_ALL) {
  const int tid = threadIdx.x;
  const int start = c * CHUNK;
  const int cnt = min(CHUNK, V - start);
  uint32_t *keys = sm.u.ch.keys;
  if (!prestaged) stage_chunk(row, start, cnt, keys);
  if (P.lp_raw && part != PART_SELECT) {
    // raw log-softmax partials: the chunk maximum of the unprocessed logits
    // and sum exp(logit - max) = sum 2^((logit - max) log2(e))
    uint32_t km = 0;
    bool b2 = false;
    for (int i = tid; i < cnt; i += SB) {
      const uint32_t k = order_key(__uint_as_float(keys[i]), b2);
      km = k > km ? k : km;
    }
    const float rmax = key_value((uint32_t)block_max_u64(km, sm));
    const Exp2Ctx ctx = exp2_ctx(LOG2E_H, LOG2E_L, rmax);
    DF acc = {0.0f, 0.0f};
    for (int i = tid; i < cnt; i += SB)
      df_accumulate(acc, df_exp2_rel(key_value(order_key(__uint_as_float(keys[i]), b2)), ctx,
                                     sm.e2h, sm.e2l));
    const DF z = block_sum_df(df_fast_two_sum(acc.h, acc.l), sm);
    if (tid == 0) {
      rec->rmax = rmax;
      rec->rzh = z.h;
      rec->rzl = z.l;
    }
  }
  if (part == PART_NORM && !P.need_z) return;
  const bool pen_on = P.n_pen > 0;
  uint32_t *penbits = sm.u.ch.penbits;
  if (pen_on) {
    // the penalty window's tokens that fall in this chunk, as a bitmap
    // (a token repeated in the window is penalised once)
    for (int w = tid; w < CHUNK / 32; w += SB) penbits[w] = 0u;
    __syncthreads();
    for (int i = tid; i < P.n_pen; i += SB) {
      const int32_t t = pen_token(P, i);
      if (t >= start && t < start + cnt)
        atomicOr(&penbits[(t - start) >> 5], 1u << ((t - start) & 31));
    }
    __syncthreads();
    if (pbits != nullptr)
      for (int w = tid; w < (cnt + 31) / 32; w += SB) pbits[c * (CHUNK / 32) + w] = penbits[w];
  }
  // the order keys, in place, and the thread's largest: four per thread at
  // a time (16-byte shared-memory accesses), then the tail
  uint32_t m = 0;
  const int nq = cnt >> 2;
  uint4 *k4 = reinterpret_cast<uint4 *>(keys);
  if (!pen_on) {
    uint32_t kmin = 0xffffffffu;
#pragma unroll 2
    for (int q = tid; q < nq; q += SB) {
      uint4 u = k4[q];
      u.x = fast_key(u.x);
      u.y = fast_key(u.y);
      u.z = fast_key(u.z);
      u.w = fast_key(u.w);
      k4[q] = u;
      const uint32_t a = u.x > u.y ? u.x : u.y, b = u.z > u.w ? u.z : u.w;
      const uint32_t c2 = u.x < u.y ? u.x : u.y, d2 = u.z < u.w ? u.z : u.w;
      m = max(m, max(a, b));
      kmin = min(kmin, min(c2, d2));
    }
    for (int i = 4 * nq + tid; i < cnt; i += SB) {
      const uint32_t k = fast_key(keys[i]);
      keys[i] = k;
      m = max(m, k);
      kmin = min(kmin, k);
    }
    // a NaN or +inf anywhere in the chunk: every thread repairs its part
    // (in the one-per-thread layout, once all the keys are written)
    if (__syncthreads_or(m >= KEY_POS_INF || kmin < KEY_NEG_INF)) m = keys_fix_bad(keys, cnt, err);
  } else {
    bool bad = false;
    for (int i = tid; i < cnt; i += SB) {
      float v = __uint_as_float(keys[i]);
      if ((penbits[i >> 5] >> (i & 31)) & 1u) v = penalise(v, P.pen);
      const uint32_t k = order_key(v, bad);
      keys[i] = k;
      m = k > m ? k : m;
    }
    if (bad) report(err, PKV_DEV_ERR_LOGITS);
  }
  __syncthreads();  // the keys, written four per thread, are read in other layouts below
  if (part == PART_NORM) {
    // the normaliser partial alone, relative to the chunk's largest key
    const uint32_t kmax = (uint32_t)block_max_u64(m, sm);
    const Exp2Ctx ctx = exp2_ctx(P.c2h, P.c2l, key_value(kmax));
    const DF z = chunk_exp_sum_all(keys, cnt, ctx, sm);
    if (tid == 0) {
      rec->zh = z.h;
      rec->zl = z.l;
    }
    __syncthreads();
    return;
  }
  const int nc = P.nc;
  const bool sel = P.mode == MODE_TOPK_SMALL || P.mode == MODE_TOPP_FULL;
  uint64_t top1 = 0ull;
  if (sel && nc <= SB) {
    // the keys at or above a bound that lets at least nc through, then the
    // nc largest of those in order
    uint32_t topkey;
    const uint32_t L = select_bound(m, nc, sm, &topkey);
    const int C = chunk_select_sorted(keys, cnt, start, L, nc, rec->cand, sm);
    if (C >= 0) {
      const int got = min(C, nc);
      for (int i = got + tid; i < nc; i += SB) rec->cand[i] = 0ull;
      if (tid == 0) {
        rec->ncand = got;
        rec->sorted = 1;
        // every token not given is below the bound: the nc-th candidate
        // when more passed, else the bound's key
        rec->thr = cnt > got ? (C > nc ? sm.nth : (uint64_t)L << 32) : 0ull;
      }
      top1 = sm.first;
    } else {
      chunk_radix_top(keys, start, cnt, nc, rec, sm);
    }
  } else if (sel) {
    chunk_radix_top(keys, start, cnt, nc, rec, sm);
  }
  if (top1 == 0ull) {
    // the chunk's largest composite: its largest key at its lowest id
    uint64_t best = 0ull;
    for (int i = tid; i < cnt; i += SB) {
      const uint64_t cc = composite(keys[i], start + i);
      best = cc > best ? cc : best;
    }
    top1 = block_max_u64(best, sm);
  }
  if (tid == 0) {
    rec->top1 = top1;
    if (!sel) {  // no candidates in this mode: a defined, empty list
      rec->ncand = 0;
      rec->thr = 0ull;
      rec->sorted = 1;
    }
    if (!P.need_z) rec->zh = rec->zl = 0.0f;
  }

  if (P.mode == MODE_ALL) {
    double bs;
    int bid;
    uint32_t bkey;
    chunk_gumbel_all(keys, start, cnt, P, sm, &bs, &bid, &bkey);
    if (tid == 0) {
      rec->gscore = bs;
      rec->gid = bid;
      rec->gkey = bkey;
    }
  }
  if (P.need_z && part == PART_ALL) {
    // sum over the chunk of exp(x - mx) = 2^(t - t_max), t = logit * log2(e) / T
    const Exp2Ctx ctx = exp2_ctx(P.c2h, P.c2l, key_value((uint32_t)(top1 >> 32)));
    const DF z = chunk_exp_sum_all(keys, cnt, ctx, sm);
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
__device__ __noinline__ int general_sample(const RowView &rv, int V, const RowParams &P, uint64_t top1,
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
      for (int r = tid; r < M; r += SB) sm.u.fi.a.es[r] = exp(comp_x(sm.sortbuf[r], P.temperature) - m);
      __syncthreads();
      if (tid == 0) {
        int r = 0;
        for (; r < M; ++r) {
          if (taken + r == 0 || (S < pz && (!minp || sm.u.fi.a.es[r] >= (double)P.min_p))) {
            S += sm.u.fi.a.es[r];
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

// The chunk records' headers into shared memory (one pass, every chunk at
// once): candidates, largest composite, bound, normaliser partial; and the
// candidates themselves into sm.u.fi.uni at stride R (a power of two >= nc;
// zeros past each chunk's count) when nch * R <= UNION_MAX.  Returns the
// total number of candidates; *all_sorted tells whether every chunk's list
// is in descending order.
__device__ int stage_records(const ChunkRec *recs, int nch, int nc, int R, SampSmem &sm,
                             bool *all_sorted, bool rec_smem = false) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    // warp 0: the headers of chunks lane and lane + 32, and over all chunks
    // the largest composite, the largest bound, the candidate count and
    // whether every list is in order
    uint64_t t1 = 0ull, bd = 0ull;
    int tot = 0, uns = 0;
#pragma unroll
    for (int h = 0; h < MAX_CHUNKS / 32; ++h) {
      const int c = tid + 32 * h;
      if (c < nch) {
        const ChunkRec &rc = recs[c];
        const int cn = rc.ncand, so = rc.sorted;
        const uint64_t top = rc.top1, thr = rc.thr;
        sm.cn[c] = cn;
        sm.htop[c] = top;
        sm.hthr[c] = thr;
        sm.fh[c] = rc.zh;
        sm.fl[c] = rc.zl;
        sm.csorted[c] = so;
        t1 = top > t1 ? top : t1;
        bd = thr > bd ? thr : bd;
        tot += cn;
        uns |= so == 0;
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const uint64_t a = __shfl_xor_sync(FULL_MASK, t1, off), b = __shfl_xor_sync(FULL_MASK, bd, off);
      t1 = a > t1 ? a : t1;
      bd = b > bd ? b : bd;
    }
    tot = __reduce_add_sync(FULL_MASK, tot);
    uns = __ballot_sync(FULL_MASK, uns) != 0u;
    if (tid == 0) {
      sm.s_top1 = t1;
      sm.s_bound = bd;
      sm.s_total = tot;
      sm.s_sorted = !uns;
    }
  }
  if (nch * R <= UNION_MAX && !rec_smem) {
    uint64_t *uni = sm.u.fi.uni;
    for (int i = tid; i < nch * R; i += SB) {
      const int c = i / R, k = i - c * R;  // R is a power of two
      if (k < nc)
        cp_async8(uni + i, recs[c].cand + k);
      else
        uni[i] = 0ull;
    }
    cp_async_wait_all();
  }
  __syncthreads();
  *all_sorted = sm.s_sorted != 0;
  return sm.s_total;
}



// Number of entries of the descending list l[0, len) greater than x
// (binary lifting over any length).
__device__ __forceinline__ int count_greater_n(const uint64_t *l, int len, uint64_t x) {
  int c = 0;
#pragma unroll 1
  for (int st = len > 0 ? 1 << (31 - __clz(len)) : 0; st > 0; st >>= 1)
    if (c + st <= len && l[c + st - 1] > x) c += st;
  return c;
}

// The exact order of the staged union's largest entries into sm.sortbuf.
// The union: nch descending lists at stride R in sm.u.fi.uni, sm.cn[c]
// long, list c holding tokens of chunk c.  The first min(cn[c], H + 1)
// entries of every list are merged pairwise, level after level (at level
// v the lists are the runs of 2^v chunks), each entry moving to its index
// in its own run plus its rank in the partner run (a binary search); the
// two buffers are sortbuf and sm.u.fi.mrg.  The (H + 1)-th entry of a
// longer list is a sentinel: below the smallest final position m* of a
// sentinel the merged order is the union's: sortbuf[0, min(m*, entries
// merged)) is exact, and that count is returned.  nch * (H + 1) <=
// GEN_BLOCK.
__device__ __noinline__ int merge_heads(int nch, int R, int H, SampSmem &sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  const uint64_t *uni = sm.u.fi.uni;
  // the heads' lengths and offsets in list order (warp 0: lists lane and lane + 32)
  if (tid < 32) {
    int h0 = lane < nch ? min(sm.cn[lane], H + 1) : 0;
    int h1 = lane + 32 < nch ? min(sm.cn[lane + 32], H + 1) : 0;
    int i0 = h0, i1 = h1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o0 = __shfl_up_sync(FULL_MASK, i0, off), o1 = __shfl_up_sync(FULL_MASK, i1, off);
      if (lane >= off) {
        i0 += o0;
        i1 += o1;
      }
    }
    const int t0 = __shfl_sync(FULL_MASK, i0, 31);
    if (lane < nch) sm.coff[lane] = i0 - h0;
    if (lane + 32 < nch) sm.coff[lane + 32] = t0 + i1 - h1;
    if (lane == 31) sm.cnt = (uint32_t)(t0 + i1);
    if (lane == 0) sm.done = 0x7fffffff;
  }
  __syncthreads();
  const int total = (int)sm.cnt;
  // offset of list c's heads (the total past the last list)
  auto offat = [&](int c) -> int { return c < nch ? sm.coff[c] : total; };
  int levels = 0;
  while ((1 << levels) < nch) ++levels;
  // start in the buffer that makes the last level write sortbuf
  uint64_t *X = (levels & 1) ? sm.u.fi.mrg : sm.sortbuf;
  uint64_t *Y = (levels & 1) ? sm.sortbuf : sm.u.fi.mrg;
  const int per = H + 1;
#pragma unroll 1
  for (int i = tid; i < nch * per; i += SB) {
    const int c = i / per, k = i - c * per;
    if (k < min(sm.cn[c], per)) X[sm.coff[c] + k] = uni[c * R + k];
  }
  __syncthreads();
#pragma unroll 1
  for (int v = 0; v < levels; ++v) {
#pragma unroll 1
    for (int g = tid; g < total; g += SB) {
      const uint64_t x = X[g];
      const int L = (comp_token(x) >> 13) >> v, P = L ^ 1;
      const int sL = offat(L << v), sP = offat(min(P << v, nch));
      const int eP = offat(min((P + 1) << v, nch));
      Y[min(sL, sP) + (g - sL) + count_greater_n(X + sP, eP - sP, x)] = x;
    }
    __syncthreads();
    uint64_t *t = X;
    X = Y;
    Y = t;
  }
  // the sentinels' final positions
  if (tid < nch && sm.cn[tid] > per - 1) {
    const int pos = count_greater_n(sm.sortbuf, total, uni[tid * R + H]);
    atomicMin(&sm.done, pos);
  }
  __syncthreads();
  const int exact = min(total, (int)sm.done);
  __syncthreads();
  return exact;
}

// The whole union in descending order into sm.u.fi.uni[0, P), P = E * SB:
// the nch lists there at stride R (a power of two, R >= E), each in
// descending order and sm.cn[c] long, padded with zeros (which order last)
// past each list and past the last list, then runs of R, 2R, ... merged
// pairwise by bitonic merging: a stage that compares entry j of a run with
// entry 2n - 1 - j of the pair (n the run length; the partner of entry i
// is i ^ (2n - 1)), then stages at distances d = n/2, ..., 1 within each
// half (partner i ^ d).  Thread t holds entries tE .. tE + E - 1 in
// registers: distances below E are compare-exchanges in the thread, those
// within the warp's 32E entries shuffles, longer ones go through shared
// memory (the two halves of sm.u.fi.uni in turn, so that one barrier per
// stage suffices).  nch * R <= P.
template <int E>
__device__ __noinline__ void bitonic_union(int nch, int R, SampSmem &sm) {
  static_assert(E == 2 || E == 4, "two or four entries a thread");
  constexpr int P = E * SB, WSPAN = 32 * E;
  static_assert(2 * P <= UNION_MAX, "two stage buffers fit the union buffer");
  uint64_t *buf = sm.u.fi.uni;
  const int tid = threadIdx.x;
  const int lr = 31 - __clz(R);
  const int b0 = tid * E;
  uint64_t v[E];
  auto load_e = [&](const uint64_t *src, uint64_t (&w)[E]) {
#pragma unroll
    for (int h = 0; h < E / 2; ++h) {
      const ulonglong2 q = reinterpret_cast<const ulonglong2 *>(src)[h];
      w[2 * h] = q.x;
      w[2 * h + 1] = q.y;
    }
  };
  auto store_e = [&](uint64_t *dst) {
#pragma unroll
    for (int h = 0; h < E / 2; ++h) {
      ulonglong2 q;
      q.x = v[2 * h];
      q.y = v[2 * h + 1];
      reinterpret_cast<ulonglong2 *>(dst)[h] = q;
    }
  };
  // the larger of the pair to the lower index
  auto keep = [](uint64_t a, uint64_t b, bool lower) -> uint64_t {
    return (lower == (b > a)) ? b : a;
  };
  load_e(buf + b0, v);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = b0 + e, c = i >> lr;
    if (c >= nch || (i & (R - 1)) >= sm.cn[c]) v[e] = 0ull;
  }
  int half = 1;  // the stage buffer the next stage through shared memory uses
#pragma unroll 1
  for (int n = R; n < P; n <<= 1) {
    const bool lo = (b0 & n) == 0;  // this thread's entries are in the first run of the pair
    uint64_t y[E];
    if (2 * n <= WSPAN) {
      const int m = (2 * n - 1) / E;  // the partner thread: lane ^ m, entry E - 1 - e
#pragma unroll
      for (int e = 0; e < E; ++e) y[e] = __shfl_xor_sync(FULL_MASK, v[E - 1 - e], m);
    } else {
      uint64_t *st = buf + half * P;
      store_e(st + b0);
      __syncthreads();
      uint64_t w[E];
      load_e(st + (b0 ^ (2 * n - E)), w);  // the partner's entries, in reverse
#pragma unroll
      for (int e = 0; e < E; ++e) y[e] = w[E - 1 - e];
      half ^= 1;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = keep(v[e], y[e], lo);
#pragma unroll 1
    for (int d = n >> 1; d >= E; d >>= 1) {
      const bool dl = (b0 & d) == 0;
      if (d < WSPAN) {
#pragma unroll
        for (int e = 0; e < E; ++e) y[e] = __shfl_xor_sync(FULL_MASK, v[e], d / E);
      } else {
        uint64_t *st = buf + half * P;
        store_e(st + b0);
        __syncthreads();
        load_e(st + (b0 ^ d), y);
        half ^= 1;
      }
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = keep(v[e], y[e], dl);
    }
    // distances below E, in the thread
#pragma unroll
    for (int dd = E / 2; dd >= 1; dd >>= 1)
#pragma unroll
      for (int e = 0; e < E; ++e)
        if ((e & dd) == 0) {
          const uint64_t a = v[e], b = v[e + dd];
          v[e] = a > b ? a : b;
          v[e + dd] = a > b ? b : a;
        }
  }
  __syncthreads();  // the last stage through shared memory may have read buf[0, P)
  store_e(buf + b0);
  __syncthreads();
}

// The nv largest composites of the union in descending order into
// sm.sortbuf[0, nv) (nv <= NCAND), read from the records in global memory:
// a radix select of the nv-th, the gather, a bitonic sort.
__device__ __noinline__ void union_sorted_slow(const ChunkRec *recs, int nc, int nu, int nv,
                                               SampSmem &sm) {
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
// partials z_c (relative to each chunk's maximum; staged in sm.fh / sm.fl)
// times 2^(t_c - t_0), added by warp 0 in a fixed order (chunks c and
// c + 32 per lane, then a xor tree).
__device__ DF row_normaliser(int nch, const Exp2Ctx &ctx, SampSmem &sm) {
  const int tid = threadIdx.x;
  DF f = {0.0f, 0.0f};
  if (tid < nch && sm.htop[tid] != 0ull) {
    const DF w = df_exp2_rel(key_value((uint32_t)(sm.htop[tid] >> 32)), ctx, sm.e2h, sm.e2l);
    f = df_mul(DF{sm.fh[tid], sm.fl[tid]}, w);
  }
  // warp 0 adds the (at most 64) rescaled partials: lanes c and c + 32,
  // then a xor tree
  __syncthreads();
  if (tid >= 32 && tid < nch) {
    sm.fh[tid] = f.h;
    sm.fl[tid] = f.l;
  }
  __syncthreads();
  if (tid < 32) {
    DF z = f;
    if (tid + 32 < nch) z = df_add(z, DF{sm.fh[tid + 32], sm.fl[tid + 32]});
#pragma unroll
    for (int off = 16; off; off >>= 1) z = df_add(z, df_shfl_xor(z, off));
    if (tid == 0) {
      sm.zh = z.h;
      sm.zl = z.l;
    }
  }
  __syncthreads();
  const DF z = {sm.zh, sm.zl};
  __syncthreads();
  return z;
}

// The first rank r in [1, n) with e_r < min_p, or n (all threads).
__device__ int minp_boundary(int n, float min_p, SampSmem &sm) {
  const DecideScratch &d = sm.u.fi.a.d;
  int first = n;
  for (int r = 1 + (int)threadIdx.x; r < n; r += SB)
    if ((d.eh[r] < min_p || (d.eh[r] == min_p && d.el[r] < 0.0f)) && r < first) first = r;
  first = __reduce_min_sync(FULL_MASK, first);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.wi[threadIdx.x >> 5] = first;
  __syncthreads();
  int m = sm.wi[0];
  for (int w = 1; w < SB / 32; ++w) m = sm.wi[w] < m ? sm.wi[w] : m;
  __syncthreads();
  return m;
}

// Sum of e_r over ranks [0, n) in a fixed order (each thread its ranks in
// order, then a xor tree per warp, then the warps in order); all threads.
__device__ DF mass_of_prefix(int n, SampSmem &sm) {
  const DecideScratch &d = sm.u.fi.a.d;
  DF part = {0.0f, 0.0f};
  for (int r = threadIdx.x; r < n; r += SB) part = df_add(part, DF{d.eh[r], d.el[r]});
  return block_sum_df(part, sm);
}

// Top-p over ranks [0, n), n <= SB * 2: rank r is kept iff r == 0 or the
// sum of the e's before it is below pz.  Each warp scans its 64 ranks
// (double-float prefix sums by shuffles), the warps' totals give each its
// carry, and the first rank not kept is the smallest over the warps.
// Returns it, or n (all threads).
__device__ int topp_cut_block(int n, DF pz, SampSmem &sm) {
  const DecideScratch &d = sm.u.fi.a.d;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r0 = warp * 64;
  DF inc[2];
  DF tot = {0.0f, 0.0f};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = r0 + 32 * h + lane;
    DF v = r < n ? DF{d.eh[r], d.el[r]} : DF{0.0f, 0.0f};
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const DF o = df_shfl_up(v, off);
      if (lane >= off) v = df_add(v, o);
    }
    inc[h] = df_add(tot, v);  // inclusive prefix within the warp's 64 ranks
    tot = df_add(tot, df_shfl(v, 31));
  }
  __syncthreads();
  if (lane == 0) {
    sm.wh[warp] = tot.h;
    sm.wl[warp] = tot.l;
  }
  __syncthreads();
  DF carry = {0.0f, 0.0f};
  for (int w = 0; w < warp; ++w) carry = df_add(carry, DF{sm.wh[w], sm.wl[w]});
  int first = n;
  const DF end0 = df_shfl(inc[0], 31);  // the prefix through the first 32 ranks
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = r0 + 32 * h + lane;
    // the sum before rank r: the carry plus the inclusive prefix of rank r - 1
    DF prev = df_shfl_up(inc[h], 1);
    if (lane == 0) prev = h == 0 ? DF{0.0f, 0.0f} : end0;
    const DF before = df_add(carry, prev);
    if (r < n && r > 0 && !df_lt(before, pz) && r < first) first = r;
  }
  first = __reduce_min_sync(FULL_MASK, first);
  __syncthreads();
  if (lane == 0) sm.wi[warp] = first;
  __syncthreads();
  int m = sm.wi[0];
  for (int w = 1; w < SB / 32; ++w) m = sm.wi[w] < m ? sm.wi[w] : m;
  __syncthreads();
  return m;
}

// Gumbel-max over the kept ranks [0, kept) of the sorted candidates s,
// whose fp32 noise is in sm's g32 for ranks below SB (computed here for the
// others): the fp32 screen, then fp64 scores for the contenders within the
// margin (see the arithmetic note above).  Returns the composite of the
// winner.
__device__ uint64_t gumbel_argmax_sorted(const uint64_t *srt, const RowParams &P, int kept,
                                         SampSmem &sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  DecideScratch &d = sm.u.fi.a.d;
  if (kept == 1) return srt[0];
  float bs = -INFINITY;
  uint64_t bc = 0ull;
  for (int r = tid; r < kept; r += SB) {
    const uint64_t cc = srt[r];
    const float g = r < SB ? d.g32[r] : gumbel32(P, comp_token(cc));
    const float s = __fadd_rn(__fdiv_rn(key_value((uint32_t)(cc >> 32)), P.temperature), g);
    d.s32[r] = s;
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
  // the screen decides unless a kept rank other than the best lies within
  // the margin (the best itself always does)
  bool other = false;
  for (int r = tid; r < kept; r += SB)
    other = other || (d.s32[r] >= floor_s && srt[r] != bestc);
  const bool screened = isfinite(best) && !__syncthreads_or(other);
  if (screened) return bestc;
  // fp64 scores of the contenders (every kept rank when the screen cannot
  // decide at all)
  const bool all = !isfinite(best);
  double ds = 0.0;
  int did = -1;
  for (int r = tid; r < kept; r += SB) {
    if (all || d.s32[r] >= floor_s) {
      const uint64_t cc = srt[r];
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
    if (comp_token(srt[r]) == id) sm.red_u64[0] = srt[r];
  __syncthreads();
  const uint64_t c = sm.red_u64[0];
  __syncthreads();
  return c;
}

// The decision over a top-k of at most 64 sorted ranks srt[0, n): every
// thread of the block takes one rank's exponential e_r and fp32 noise first
// (into DecideScratch), then warp 0 alone decides with shuffles and ballots
// (no further block barrier but the last), lane l holding ranks 2l and
// 2l + 1: min_p (the first rank >= 1 with e_r < min_p), top-p (one
// double-float scan over the lanes' pair sums; Z is its total), the Gumbel
// argmax (the fp32 screen, fp64 for the contenders within its margin).
// A row takes this path or the block-wide one by its own settings alone.
// With log-probs requested, also leaves sm.s_kept, sm.m_row and sm.xbest.
// Returns the winner's composite (all threads).
__device__ __noinline__ uint64_t decide_small(const uint64_t *srt, int n, const RowParams &P,
                                              const Exp2Ctx &ctx, SampSmem &sm) {
  DecideScratch &d = sm.u.fi.a.d;
  for (int r = threadIdx.x; r < n; r += SB) {
    const uint64_t cc = srt[r];
    const DF e = df_exp2_rel(key_value((uint32_t)(cc >> 32)), ctx, sm.e2h, sm.e2l);
    d.eh[r] = e.h;
    d.el[r] = e.l;
    d.g32[r] = gumbel32(P, comp_token(cc));
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const DF zero = {0.0f, 0.0f};
    const int r0 = 2 * lane, r1 = 2 * lane + 1;
    const bool v0 = r0 < n, v1 = r1 < n;
    const uint64_t c0 = v0 ? srt[r0] : 0ull, c1 = v1 ? srt[r1] : 0ull;
    const DF e0 = v0 ? DF{d.eh[r0], d.el[r0]} : zero;
    const DF e1 = v1 ? DF{d.eh[r1], d.el[r1]} : zero;
    // min_p: the first rank >= 1 with e_r < min_p
    int kp = n;
    if (P.min_p > 0.0f) {
      const bool cut0 = r0 >= 1 && v0 && (e0.h < P.min_p || (e0.h == P.min_p && e0.l < 0.0f));
      const bool cut1 = v1 && (e1.h < P.min_p || (e1.h == P.min_p && e1.l < 0.0f));
      kp = __reduce_min_sync(FULL_MASK, cut0 ? r0 : (cut1 ? r1 : n));
    }
    // top-p over ranks [0, kp): rank r is kept iff r == 0 or the sum of the
    // e's before it is below p * Z
    int kept = kp;
    if (P.top_p < 1.0f) {
      const DF a0 = r0 < kp ? e0 : zero, a1 = r1 < kp ? e1 : zero;
      const DF pair = df_add(a0, a1);
      DF incl = pair;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const DF o = df_shfl_up(incl, off);
        if (lane >= off) incl = df_add(o, incl);
      }
      const DF pz = df_mul_f(df_shfl(incl, 31), P.top_p);
      DF before0 = df_shfl_up(incl, 1);  // the sum over ranks < r0
      if (lane == 0) before0 = zero;
      const DF before1 = df_add(before0, a0);
      int first = kp;
      if (r1 < kp && !df_lt(before1, pz)) first = r1;
      if (r0 >= 1 && r0 < kp && !df_lt(before0, pz)) first = r0;
      kept = __reduce_min_sync(FULL_MASK, first);
    }
    // Gumbel-max over ranks [0, kept): the fp32 screen, fp64 for contenders
    uint64_t win = __shfl_sync(FULL_MASK, c0, 0);
    if (kept > 1) {
      const float s0 = r0 < kept
                           ? __fadd_rn(__fdiv_rn(key_value((uint32_t)(c0 >> 32)), P.temperature), d.g32[r0])
                           : -INFINITY;
      const float s1 = r1 < kept
                           ? __fadd_rn(__fdiv_rn(key_value((uint32_t)(c1 >> 32)), P.temperature), d.g32[r1])
                           : -INFINITY;
      // the lane's better of its two ranks (score descending, token ascending)
      float bs = -INFINITY;
      uint64_t bc = 0ull;
      if (r0 < kept) {
        bs = s0;
        bc = c0;
      }
      if (r1 < kept && (bc == 0ull || s1 > bs || (s1 == bs && comp_token(c1) < comp_token(bc)))) {
        bs = s1;
        bc = c1;
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
      const float floor_s = bs - (1e-4f + 2e-6f * fabsf(bs));
      const int close = __popc(__ballot_sync(FULL_MASK, r0 < kept && s0 >= floor_s)) +
                        __popc(__ballot_sync(FULL_MASK, r1 < kept && s1 >= floor_s));
      if (isfinite(bs) && close == 1) {
        win = bc;
      } else {
        const bool all = !isfinite(bs);
        double ds = 0.0;
        int did = -1;
        uint64_t dc = 0ull;
        if (r0 < kept && (all || s0 >= floor_s)) {
          ds = comp_x(c0, P.temperature) + gumbel(P, comp_token(c0));
          did = comp_token(c0);
          dc = c0;
        }
        if (r1 < kept && (all || s1 >= floor_s)) {
          const double v = comp_x(c1, P.temperature) + gumbel(P, comp_token(c1));
          if (better(v, comp_token(c1), ds, did)) {
            ds = v;
            did = comp_token(c1);
            dc = c1;
          }
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
          const double os = __shfl_xor_sync(FULL_MASK, ds, off);
          const int oi = __shfl_xor_sync(FULL_MASK, did, off);
          const uint64_t oc = __shfl_xor_sync(FULL_MASK, dc, off);
          if (better(os, oi, ds, did)) {
            ds = os;
            did = oi;
            dc = oc;
          }
        }
        win = dc;
      }
    }
    if (P.lp_proc) {
      // the kept ranks' mass
      DF v = df_add(r0 < kept ? e0 : zero, r1 < kept ? e1 : zero);
#pragma unroll
      for (int off = 16; off; off >>= 1) v = df_add(v, df_shfl_xor(v, off));
      if (lane == 0) {
        sm.s_kept = (double)v.h + (double)v.l;
        sm.m_row = comp_x(c0, P.temperature);
        sm.xbest = comp_x(win, P.temperature);
      }
    }
    if (lane == 0) sm.first = win;
  }
  __syncthreads();
  const uint64_t w = sm.first;
  __syncthreads();
  return w;
}

// With log-probs requested (and not greedy), leaves the kept mass relative
// to the row maximum, that maximum's x and the sampled token's x in
// sm.s_kept, sm.m_row and sm.xbest.
// rec_smem: the single chunk's record is in shared memory (its candidate
// list is read in place).
__device__ __noinline__ int finish_row(const RowView &rv, int V, int nch, const RowParams &P,
                                       const ChunkRec *recs, SampSmem &sm, bool rec_smem = false) {
  const int tid = threadIdx.x;
  const int nc = P.nc;
  int R = 1;
  while (R < nc) R <<= 1;
  bool all_sorted;
  const bool cand_mode = P.mode == MODE_TOPK_SMALL || P.mode == MODE_TOPP_FULL;
  const int nreal = stage_records(recs, nch, nc, cand_mode ? R : 0, sm, &all_sorted, rec_smem);
  const uint64_t top1 = sm.s_top1;
  // the chunks hold no token outside the union above this bound
  const uint64_t bound = sm.s_bound;
  if (P.mode == MODE_GREEDY) return comp_token(top1);
  const Exp2Ctx ctx = exp2_ctx(P.c2h, P.c2l, key_value((uint32_t)(top1 >> 32)));
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
      const DF z = row_normaliser(nch, ctx, sm);
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
  // candidates that the decision reads
  const int nu = nch * R;
  const bool full = P.mode == MODE_TOPP_FULL;
  const bool topp = P.top_p < 1.0f;
  const bool minp = P.min_p > 0.0f;
  DecideScratch &d = sm.u.fi.a.d;
  // ranks the decision may read: the top-k, or for top-p over the whole
  // vocabulary up to NCAND candidates (past them: the general path)
  const int nv = min(full ? NCAND : P.K, nreal);
  // top-p over the whole vocabulary without min_p: Z is the whole row's
  const bool z_row = full && !minp;
  DF Z = {0.0f, 0.0f};
  if (z_row) Z = row_normaliser(nch, ctx, sm);
  // The sorted prefix the decision reads: a top-k's survivors; for top-p
  // over the whole vocabulary the first 256 ranks, then, if the decision is
  // still open there, all NCAND.  A single chunk's list is in order already.
  const bool staged = nu <= UNION_MAX && all_sorted;
  const uint64_t *srt = sm.sortbuf;
  int kept = 0, kp = nv;
  bool general = true;
  const int hmax = GEN_BLOCK / nch - 1;  // longest heads that fit the merge buffers
  for (int attempt = 0; attempt < 3; ++attempt) {
    int avail = nv;
    if (nch == 1 && staged) {
      srt = rec_smem ? recs[0].cand : sm.u.fi.uni;
      attempt = 2;  // nothing more to read later
    } else if (staged && !rec_smem && R >= 4 && nch * R <= 4 * SB) {
      // the whole union in order, in place
      if (nch * R <= 2 * SB)
        bitonic_union<2>(nch, R, sm);
      else
        bitonic_union<4>(nch, R, sm);
      srt = sm.u.fi.uni;
      attempt = 2;
    } else if (staged && attempt < 2) {
      // the heads of the lists first, about twice each list's share of the
      // ranks wanted (for top-p over the whole vocabulary 256 at first),
      // then as much of them as the merge buffers hold
      int H = hmax;
      if (attempt == 0) {
        const int want = full ? min(256, nv) : nv;
        H = 8;
        while (H < hmax && H * nch < 2 * want) H <<= 1;
        H = min(H, hmax);
      }
      avail = min(nv, merge_heads(nch, R, H, sm));
      srt = sm.sortbuf;
      if (H >= nc) attempt = 2;  // the whole lists were read
    } else {
      union_sorted_slow(recs, nc, nch * nc, nv, sm);
      srt = sm.sortbuf;
      attempt = 2;
    }
    if (!full && avail < nv) continue;  // the top-k survivors are not all in order yet
    if (!full && nv <= 64) {
      // a top-k of at most 64: decided by one warp when the order is exact
      if (srt[nv - 1] >= bound && !(P.K > nreal))
        return comp_token(decide_small(srt, nv, P, ctx, sm));
      break;  // every candidate was read: the general path
    }
    // e_r = 2^(t_r - t_0) of the ranks the decision may read, and the fp32
    // noise of the first SB of them
    for (int r = tid; r < avail; r += SB) {
      const uint64_t cc = srt[r];
      const DF e = df_exp2_rel(key_value((uint32_t)(cc >> 32)), ctx, sm.e2h, sm.e2l);
      d.eh[r] = e.h;
      d.el[r] = e.l;
      if (r < SB) d.g32[r] = gumbel32(P, comp_token(cc));
    }
    __syncthreads();
    // ranks of the row past the ones read here
    const bool beyond = full && avail < V;
    // min_p, then top-p over the ranks that pass top-k and min_p
    kp = minp ? minp_boundary(avail, P.min_p, sm) : avail;
    bool open = minp && kp == avail && beyond;  // min_p boundary not reached
    kept = kp;
    if (!open && topp) {
      const DF z = z_row ? Z : mass_of_prefix(kp, sm);
      if (!z_row) Z = z;
      kept = topp_cut_block(kp, df_mul_f(z, P.top_p), sm);
      if (kept == kp && !minp && beyond) open = true;  // top-p not reached
    }
    // The sorted prefix is the exact global order over the ranks the
    // decision read (the kept set; the ranks through the min_p boundary;
    // for top-k the K survivors) when its last one is at or above the
    // bound under which the chunks hold tokens not in the union.  The top-k
    // also needs K candidates in the union.
    bool exact = !open;
    if (exact) {
      const int decided = !full ? nv : (minp ? min(kp + 1, avail) : kept);
      exact = srt[decided - 1] >= bound && !(!full && P.K > nreal);
    }
    if (exact) {
      general = false;
      break;
    }
    if (avail == nv) break;  // every candidate was read
  }
  if (general) {
    const double zk = z_row ? (double)Z.h + (double)Z.l : -1.0;
    return general_sample(rv, V, P, top1, zk, sm);
  }
  const uint64_t win = gumbel_argmax_sorted(srt, P, kept, sm);
  if (P.lp_proc) {
    const DF sk = mass_of_prefix(kept, sm);
    if (tid == 0) {
      sm.s_kept = (double)sk.h + (double)sk.l;
      sm.m_row = comp_x(srt[0], P.temperature);
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
  int zsplit;      // a second CTA per chunk (grid rows B..2B-1) takes the normaliser
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

// One CTA per (chunk, row); with zsplit, grid rows B..2B-1 are a second CTA
// per chunk that computes the chunk's normaliser partial while the first
// selects the candidates (rows that need no normaliser leave it at once).
__global__ void __launch_bounds__(SB) sample_chunk_kernel(const SampleArgs a) {
  __shared__ SampSmem sm;
  const bool zcta = (int)blockIdx.y >= a.batch;
  const int b = zcta ? (int)blockIdx.y - a.batch : (int)blockIdx.y;
  const int c = blockIdx.x;
  // launched behind its predecessor on the stream (programmatic dependent
  // launch): nothing is read before that grid has completed
  pdl_wait();
  // The finish kernel may be scheduled once every chunk CTA has passed this
  // point (or exited), so once the last chunk CTA has started: its CTAs
  // then take only the room that chunk CTAs leave, and have their prologue
  // done when the last chunk CTA ends.
  pdl_trigger();
  if (!a.active[b]) return;
  const int slot = a.slots[b];
  if (slot < 0 || slot >= a.num_slots) return;
  RowParams P;
  if (zcta) {
    // a second CTA: only when the row asks for a normaliser
    P = sample_row_params(a, slot);
    if (!(P.need_z || P.lp_raw)) return;
  }
  // the chunk's copies go out first; the row's parameters are formed while
  // they are in flight
  const float *row = a.logits + (int64_t)b * a.row_stride;
  const bool bulk = stage_chunk_begin(row, c * CHUNK, min(CHUNK, a.vocab - c * CHUNK), sm);
  if (!zcta) P = sample_row_params(a, slot);
  load_exp2_table(sm);
  if (!stage_chunk_end(bulk, sm, a.err)) {
    // reported; the record says "no candidates" so that the finish reads a
    // well-formed one
    ChunkRec *rec = a.recs + (int64_t)b * a.nch + c;
    if (!zcta && threadIdx.x == 0) {
      rec->ncand = 0;
      rec->sorted = 1;
      rec->top1 = 0ull;
      rec->thr = 0ull;
    }
    return;
  }
  int part = PART_ALL;
  if (a.zsplit && (P.need_z || P.lp_raw)) part = zcta ? PART_NORM : PART_SELECT;
  chunk_pass(row, a.vocab, c, P, a.recs + (int64_t)b * a.nch + c,
             part == PART_NORM ? nullptr : row_pbits(a, b), sm, a.err, true, part);
}

__device__ __forceinline__ void sample_skip_row(const SampleArgs &a, int b) {
  a.out_tok[b] = 0;
  a.out_kind[b] = PKV_KIND_OTHER;
  if (a.lp_raw != nullptr) a.lp_raw[b] = 0.0f;
  if (a.lp_proc != nullptr) a.lp_proc[b] = 0.0f;
}

// The finish of row b from its chunk records (in global memory, or for a
// single-chunk row in shared memory): the decision, the log-probs, the
// outputs and the slot's step counter and ring.
__device__ __forceinline__ void finish_write(const SampleArgs &a, int b, int slot, const RowParams &P,
                                          const ChunkRec *recs, SampSmem &sm, bool rec_smem) {
  const int tid = threadIdx.x;
  const float *row = a.logits + (int64_t)b * a.row_stride;
  const RowView rv = {row, P.n_pen > 0 ? row_pbits(a, b) : nullptr, P.pen};
  const int tok = finish_row(rv, a.vocab, a.nch, P, recs, sm, rec_smem);
  double lse_raw = 0.0;
  if (P.lp_raw) {
    // log-sum-exp of the unprocessed row: the chunks' partials rescaled to
    // the row maximum in parallel, added in chunk order
    float rm = recs[0].rmax;
    for (int c = 1; c < a.nch; ++c) rm = fmaxf(rm, recs[c].rmax);
    __syncthreads();
    double *part = sm.u.fi.a.es;  // free once the decision is taken
    if (tid < a.nch)
      part[tid] = ((double)recs[tid].rzh + (double)recs[tid].rzl) *
                  exp((double)recs[tid].rmax - (double)rm);
    __syncthreads();
    if (tid == 0) {
      double z = 0.0;
      for (int c = 0; c < a.nch; ++c) z += part[c];
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

__global__ void __launch_bounds__(SB) sample_finish_kernel(const SampleArgs a) {
  __shared__ SampSmem sm;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  // This grid starts once every chunk CTA has passed its own wait for its
  // predecessors, so everything but the chunk records (the flags, the slot
  // settings and step counters, the history ring) is final already: read it
  // before waiting for the chunk records.
  const int active = a.active[b];
  const int slot = a.slots[b];
  const bool ok = active && slot >= 0 && slot < a.num_slots;
  RowParams P;
  if (ok) P = sample_row_params(a, slot);
  load_exp2_table(sm);  // read after finish_row's first barrier
  pdl_wait();  // the chunk records
  if (!ok) {
    if (tid == 0) {
      sample_skip_row(a, b);
      if (active) report(a.err, PKV_DEV_ERR_SLOT);
    }
    return;
  }
  finish_write(a, b, slot, P, a.recs + (int64_t)b * a.nch, sm, false);
}

// A vocabulary of one chunk: one CTA per row runs the chunk pass and the
// finish, with the chunk record in the part of the shared union the keys
// leave free when the row has at most SREC_MAX_V tokens (else in the
// workspace): the same arithmetic as the two kernels, without the second
// launch and the records' round trip.
__global__ void __launch_bounds__(SB) sample_single_kernel(const SampleArgs a) {
  __shared__ SampSmem sm;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const int active = a.active[b];
  const int slot = a.slots[b];
  if (!active || slot < 0 || slot >= a.num_slots) {
    if (tid == 0) {
      sample_skip_row(a, b);
      if (active) report(a.err, PKV_DEV_ERR_SLOT);
    }
    return;
  }
  const RowParams P = sample_row_params(a, slot);
  load_exp2_table(sm);  // read after the first barrier of the chunk pass
  const bool rs = a.vocab <= SREC_MAX_V;
  ChunkRec *rec = rs ? reinterpret_cast<ChunkRec *>(sm.u.fi.mrg) : a.recs + (int64_t)b * a.nch;
  chunk_pass(a.logits + (int64_t)b * a.row_stride, a.vocab, 0, P, rec, row_pbits(a, b), sm,
             a.err);
  __syncthreads();
  finish_write(a, b, slot, P, rec, sm, rs);
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
  // A single-chunk row of up to SREC_MAX_V tokens keeps its record in the
  // part of the shared union that its keys leave free (the merge buffer,
  // which a single chunk's finish does not use): no round trip through
  // global memory between the chunk pass and the finish.
  ChunkRec *srec = reinterpret_cast<ChunkRec *>(sm.u.fi.mrg);
  if (a.ctrl != nullptr) {
    // channel 0: the stop/continue sample (salt 0); a stop ends the frame
    const float *crow = a.ctrl + (int64_t)b * a.ctrl_vocab;
    const RowParams P = row_params(a.ctrl_vocab, a.seeds[slot], step, a.temperature[slot],
                                   a.top_k[slot], a.top_p[slot], 0u);
    const bool cs = a.ctrl_nch == 1 && a.ctrl_vocab <= SREC_MAX_V;
    ChunkRec *cr = cs ? srec : recs;
    for (int c = 0; c < a.ctrl_nch; ++c) {
      chunk_pass(crow, a.ctrl_vocab, c, P, cr + c, nullptr, sm, a.err);
      __syncthreads();
    }
    const int tok =
        finish_row(RowView{crow, nullptr, 1.0f}, a.ctrl_vocab, a.ctrl_nch, P, cr, sm, cs);
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
    bool prestaged = false;
    if (j > 0 && a.fb != nullptr) {
      // base[j] + fb[j][code_{j-1}], rounded once to fp32: into the chunk
      // buffer directly when the row is one chunk, and to the row buffer in
      // global memory (which the general path and longer rows read)
      const float *f = a.fb + ((int64_t)j * V + prev) * V;
      prestaged = V <= CHUNK;
      for (int i = tid; i < V; i += SB) {
        const float v = __fadd_rn(row[i], f[i]);
        rowbuf[i] = v;
        if (prestaged) sm.u.ch.keys[i] = __float_as_uint(v);
      }
      __threadfence_block();
      __syncthreads();
      row = rowbuf;
    }
    const RowParams P = row_params(V, a.seeds[slot], step, a.temperature[slot], a.top_k[slot],
                                   a.top_p[slot], (uint32_t)(1 + j));
    const bool rs = a.nch == 1 && V <= SREC_MAX_V;
    ChunkRec *rr = rs ? srec : recs;
    for (int c = 0; c < a.nch; ++c) {
      chunk_pass(row, V, c, P, rr + c, nullptr, sm, a.err, prestaged);
      __syncthreads();
    }
    const int tok = finish_row(RowView{row, nullptr, 1.0f}, V, a.nch, P, rr, sm, rs);
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

// Chunk CTAs resident at once on the current device (SMs x CTAs per SM; 0
// when it cannot be read); cached per device
static int chunk_ctas_resident() {
  static std::atomic<int> count[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int n = count[dev & 63].load(std::memory_order_relaxed);
  if (n == 0) {
    int sms = 0, per = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, pkv::sample_chunk_kernel, pkv::SB, 0) !=
            cudaSuccess)
      return 0;
    n = sms * per;
    count[dev & 63].store(n, std::memory_order_relaxed);
  }
  return n;
}

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
  // a second CTA per chunk for the normaliser when the two fit on the SMs
  // at once
  const int64_t resident = chunk_ctas_resident();
  if (resident <= 0) return PKV_ERR_CUDA;
  const int64_t ctas = (int64_t)a.nch * batch;
  a.zsplit = 2 * ctas <= resident ? 1 : 0;
  if (a.nch == 1) {
    // one chunk a row: chunk pass and finish in one CTA
    if (launch_pdl(sample_single_kernel, dim3((unsigned)batch), dim3(SB), 0, s, a) != cudaSuccess)
      return PKV_ERR_CUDA;
    return launch_status();
  }
  if (launch_pdl(sample_chunk_kernel, dim3((unsigned)a.nch, (unsigned)(batch * (1 + a.zsplit))),
                 dim3(SB), 0, s, a) != cudaSuccess)
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
