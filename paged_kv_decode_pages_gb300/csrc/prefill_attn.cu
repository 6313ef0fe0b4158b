// prefill_attn.cu -- causal attention of a step's new tokens over the paged
// cache: prompt rows of a prefill ("Adding a Model", vox-serve docs, "How a
// program runs": lm_prefill over row buckets) and mixed steps that carry
// decode rows beside prompt rows ("Supported Models", mstar docs, Qwen3.5 /
// Qwen3.8 notes).  Request b's q_b new tokens (packed rows qo_indptr[b] ..
// qo_indptr[b+1]) sit at positions seq_len - q_b .. seq_len - 1, already
// appended to the cache; the token at position p attends to positions
// [0, p] of its request.
//
// This is a dense contraction, so it runs on the 5th-generation tensor
// cores:
//  * a q tile is 128 MMA rows: tq = 128 / G tokens x the G q heads of one
//    kv head (GQA packing: every K / V tile read serves the whole group);
//  * one CTA per (request, pair of consecutive q tiles, kv head): the two
//    tiles share every K / V tile, and while one tile's softmax runs on the
//    CUDA cores the tensor cores work on the other's products; a one-CTA
//    planner lists the pairs (prefix sums), requests with the longest
//    context first and the heaviest pair of each request first;
//  * a K load warp (both tiles' Q once, then the K tiles) and a V load warp
//    bring 128-key tiles (16-token blocks of the pages, or 128-row boxes on
//    128-token pages; 128-byte swizzle) into shared memory by tiled tensor
//    TMA; an MMA warp issues, per KV tile, S = Q K^T of both tiles into
//    tensor memory and then O += P V of both (bf16 operands, fp32
//    accumulation in tensor memory), each completion signalled by
//    tcgen05.commit on an mbarrier.  Tensor memory holds S and O of both
//    tiles (all 512 columns), so P goes through shared memory;
//  * two softmax warpgroups, one per tile, own one row per thread: they
//    read the row of S from tensor memory, apply the causal mask, run the
//    online softmax in log2 units with a lazy maximum (O is rescaled in
//    tensor memory only when the running maximum grows by more than 8),
//    write P as bf16 into shared memory in the swizzled K-major layout of
//    the A operand, and at the end read O, divide by the row sum and store
//    it;
//  * stale cache slots past a request's last position are zeroed in shared
//    memory before they meet P (whose entries there are 0), so whatever an
//    unwritten slot holds cannot reach the output;
//  * every wait is bounded; a give-up is reported and the CTA drains its
//    tensor-core work before it frees its tensor memory.
#include <math.h>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int PF_M = 128;          // MMA rows of a tile
constexpr int PF_N = 128;          // keys of a KV tile
constexpr int PF_BLK = 16;         // tokens of one cache block (one TMA box)
constexpr int PF_SM_WARPS = 8;     // two softmax warpgroups, one per q tile of the unit
constexpr int PF_THREADS = 384;    // + K load warp, tile A's MMA warp, V load warp, tile B's MMA warp
constexpr int PF_CHUNK = 16384;    // 128 rows x 128 bytes (64 bf16): one swizzle column
constexpr int PF_TMEM_COLS = 512;  // S of both tiles (128 columns each), O of both (128 each)
constexpr int PF_PLAN_THREADS = 1024;
constexpr float PF_TAU = 8.0f;     // lazy-rescale threshold (log2 units)

struct PfHeader {
  int32_t total_pairs;
  int32_t total_units;
  int32_t pad_[2];
};

struct PfArgs {
  int layer;
  int num_pages;
  int bpp;  // 16-token blocks per page
  int num_kv_heads;
  int num_qo_heads;
  int group;
  int tq;   // tokens per tile
  int T;
  float qscale;  // sm_scale * log2(e)
  const int32_t *qo_indptr;
  const int32_t *page_table;
  int max_pages;
  int64_t max_tokens;
  const int32_t *seq_lens;
  const int32_t *active;
  int batch;
  uint16_t *out;  // bf16 [T][Hq][D]
  float *lse;     // [T][Hq] or null
  int32_t *tile_start;  // [B + 1] first unit (pair of q tiles) of each position of the schedule
  int32_t *order;       // [B] request at each position (longest context first)
  PfHeader *hdr;
  int32_t *err;
};

// ---------------------------------------------------------------------------
// tcgen05 / tensor-memory wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle.  K-major operands: rows
// of 128 bytes, 8-row groups 1024 bytes apart (sbo); the leading offset is
// not used.  MN-major operands: lbo = distance between 64-element atoms
// along MN, sbo = distance between 8-row groups along K.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version of the 5th-generation tensor cores
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, A
// K-major, B K-major or MN-major, M x N.
__host__ __device__ constexpr uint32_t bf16_idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 32 consecutive 32-bit columns of the warp's 32 lanes
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, int c0, int c1, int c2,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  return *reinterpret_cast<const uint32_t *>(&v);
}

// ---------------------------------------------------------------------------
// planner: one CTA lists the units (pairs of q tiles) of every request
// (prefix sums)
// ---------------------------------------------------------------------------
// units of a request: pairs of its q tiles (the last unit of an odd count
// holds one tile)
__device__ __forceinline__ int request_units(const PfArgs &a, int b) {
  const int q = a.qo_indptr[b + 1] - a.qo_indptr[b];
  return q > 0 ? ((q + a.tq - 1) / a.tq + 1) / 2 : 0;
}

// schedule key of a request: its context length (the KV its heaviest tile
// streams), -1 when it has no tiles
__device__ __forceinline__ int request_key(const PfArgs &a, int b) {
  const int q = a.qo_indptr[b + 1] - a.qo_indptr[b];
  if (q <= 0) return -1;
  const int n = a.seq_lens[b];
  return n > 0 ? n : 0;
}

__global__ void __launch_bounds__(PF_PLAN_THREADS) prefill_plan_kernel(const PfArgs a) {
  __shared__ int32_t scan[PF_PLAN_THREADS];
  __shared__ int32_t carry;
  pdl_trigger();
  const int tid = threadIdx.x;
  if (tid == 0) carry = 0;
  // the schedule: requests by descending context length (ties by index), so
  // that the longest units start first and the short ones fill the tail
  for (int b = tid; b < a.batch; b += PF_PLAN_THREADS) {
    if (a.qo_indptr[b + 1] < a.qo_indptr[b] || (b == 0 && a.qo_indptr[0] != 0))
      report(a.err, PKV_DEV_ERR_INDPTR);
    const int kb = request_key(a, b);
    int rank = 0;
    for (int o = 0; o < a.batch; ++o) {
      const int ko = request_key(a, o);
      rank += (ko > kb || (ko == kb && o < b)) ? 1 : 0;
    }
    a.order[rank] = b;
  }
  __syncthreads();
  for (int base = 0; base < a.batch; base += PF_PLAN_THREADS) {
    const int i = base + tid;
    int nt = 0;
    if (i < a.batch) {
      const int b = a.order[i];
      if (a.qo_indptr[b + 1] >= a.qo_indptr[b]) nt = request_units(a, b);
    }
    scan[tid] = nt;
    __syncthreads();
    for (int off = 1; off < PF_PLAN_THREADS; off <<= 1) {
      const int v = tid >= off ? scan[tid - off] : 0;
      __syncthreads();
      scan[tid] += v;
      __syncthreads();
    }
    if (i < a.batch) a.tile_start[i] = carry + scan[tid] - nt;
    __syncthreads();
    if (tid == PF_PLAN_THREADS - 1) carry += scan[tid];
    __syncthreads();
  }
  if (tid == 0) {
    a.tile_start[a.batch] = carry;
    a.hdr->total_pairs = carry;
    a.hdr->total_units = carry * a.num_kv_heads;
    if (a.qo_indptr[a.batch] > a.T) report(a.err, PKV_DEV_ERR_INDPTR);
  }
  pdl_wait();  // completes after the append that wrote the step's tokens
}

// ---------------------------------------------------------------------------
// the attention kernel
// ---------------------------------------------------------------------------
template <int D>
struct PfShape {
  static constexpr int NCH = D / 64;                  // 64-dim swizzle columns
  static constexpr int TILE_BYTES = NCH * PF_CHUNK;   // a Q tile, or one K / V stage
  static constexpr int P_BYTES = 2 * PF_CHUNK;        // P: 128 rows x 128 keys
  static constexpr int NK = 2;                        // K stages
  static constexpr int NV = D == 64 ? 2 : 1;          // V stages (head_dim 128: the space
                                                      // is taken by the two tiles' Q and P)
  static constexpr int OFF_Q = 0;                     // [2 tiles]
  static constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NK * TILE_BYTES;
  static constexpr int OFF_P = OFF_V + NV * TILE_BYTES;  // [2 tiles]
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr int NBAR = 19;
  // + alignment slack; at least 120 KB, so that one CTA (which holds all
  // 512 tensor-memory columns) is resident per SM
  static constexpr int RAW = OFF_BAR + NBAR * 8 + 16 + 1024;
  static constexpr int SMEM_BYTES = RAW > 120 * 1024 ? RAW : 120 * 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// One tile of a unit: its tokens, their positions and the KV tiles they read.
struct PfTile {
  int t0;    // first packed row
  int ntok;  // tokens (0: no tile)
  int pos0;  // position of the first token
  int nkv;   // 128-key tiles read (0: no tile)
};

template <int D>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_attn_kernel(const PfArgs a, const __grid_constant__ CUtensorMap kv_map,
                        const __grid_constant__ CUtensorMap kv_map128,
                        const __grid_constant__ CUtensorMap q_map) {
  using S = PfShape<D>;
  constexpr int NCH = S::NCH, NV = S::NV;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char *qs = sm + S::OFF_Q;  // [2 tiles][NCH][128 rows][128 B]
  unsigned char *ks = sm + S::OFF_K;  // [NK][NCH][128 rows][128 B]
  unsigned char *vs = sm + S::OFF_V;  // [NV][NCH][128 rows][128 B]
  unsigned char *ps = sm + S::OFF_P;  // [2 tiles][2 key columns][128 rows][128 B]
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + S::OFF_BAR);
  uint64_t *bar_q = bars + 0;       // both tiles' Q
  uint64_t *bar_k = bars + 1;       // [2] K stage loaded
  uint64_t *bar_v = bars + 3;       // [2] V stage loaded
  uint64_t *bar_s = bars + 5;       // [tile] S computed
  uint64_t *bar_sfree = bars + 7;   // [tile] S read out of tensor memory by all 128 rows
  uint64_t *bar_p = bars + 9;       // [tile] P written, O rescaled (128 rows)
  uint64_t *bar_o = bars + 11;      // [tile] P.V computed
  uint64_t *bar_kfree = bars + 13;  // [2] the S products of the K stage's tile have completed
  uint64_t *bar_vfree = bars + 15;  // [2] the P.V products of the V stage's tile have completed
  uint64_t *bar_fin = bars + 17;   // both MMA warps' products have completed
  uint64_t *bar_vz = bars + 18;    // the stale V rows are zeroed (tile A's MMA warp)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + S::NBAR);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int Hkv = a.num_kv_heads;
  const int G = a.group;
  const int Hq = a.num_qo_heads;

  pdl_wait();  // the planner's table, the append's cache writes
  pdl_trigger();
  const int u = blockIdx.x;
  if (u >= a.hdr->total_units) return;
  const int su = u / Hkv, g = u % Hkv;
  // schedule position of unit su: the last i with tile_start[i] <= su
  // (tile_start is non-decreasing).  Up to 64 requests: the warp's lanes
  // test 32 positions per load; else a binary search.
  int lo = 0;
  if (a.batch <= 64) {
    for (int base = 0; base < a.batch; base += 32) {
      const int i = base + lane;
      const unsigned m = __ballot_sync(FULL_MASK, i < a.batch && a.tile_start[i] <= su);
      if (m) lo = base + 31 - __clz(m);
      if (m != FULL_MASK) break;
    }
  } else {
    int hi = a.batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.tile_start[mid] <= su)
        lo = mid;
      else
        hi = mid - 1;
    }
  }
  const int b = a.order[lo];
  const int q = a.qo_indptr[b + 1] - a.qo_indptr[b];
  const int nt = (q + a.tq - 1) / a.tq;  // q tiles of the request
  const int pi = su - a.tile_start[lo];  // pair index, heaviest first
  const int n = a.seq_lens[b];
  const bool ok = a.active[b] && q <= n && n >= 1 && (int64_t)n <= a.max_tokens;
  // tile A: the later (longer) q tile of the pair; tile B the one before it
  PfTile tl[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int ti = nt - 1 - 2 * pi - x;
    if (ti < 0) {
      tl[x] = PfTile{0, 0, 0, 0};
      continue;
    }
    tl[x].t0 = a.qo_indptr[b] + ti * a.tq;
    tl[x].ntok = min(a.tq, q - ti * a.tq);
    tl[x].pos0 = n - q + ti * a.tq;
    tl[x].nkv = ok ? (tl[x].pos0 + tl[x].ntok - 1) / PF_N + 1 : 0;
  }

  if (!ok) {
    // padding or malformed request: zeros, lse = -inf
    if (a.active[b] && pi == 0 && g == 0 && tid == 0) report(a.err, PKV_DEV_ERR_SEQ_LEN);
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int rows = tl[x].ntok * G;
      for (int r = warp; r < rows; r += PF_THREADS / 32) {
        const int t = tl[x].t0 + r / G, h = g * G + r % G;
        if (t >= a.T) break;
        uint16_t *o = a.out + ((int64_t)t * Hq + h) * D;
        for (int d = lane * 2; d < D; d += 64) *reinterpret_cast<uint32_t *>(o + d) = 0u;
        if (a.lse != nullptr && lane == 0) a.lse[(int64_t)t * Hq + h] = -INFINITY;
      }
    }
    return;
  }
  const int nkv = tl[0].nkv;               // KV tiles read by the unit (tile A reads the most)
  const int last_blk = (n - 1) / PF_BLK;   // block of the request's last position
  const int kt_stale = (n - 1) / PF_N;     // the KV tile that holds slots past n - 1

  if (tid == 0) {
    for (int i = 0; i < S::NBAR; ++i)
      // sfree, p: one arrival per row; K / V stage releases and the drain:
      // one commit per MMA warp
      mbar_init(&bars[i], (i >= 7 && i <= 10) ? 128u : ((i >= 13 && i <= 17) ? 2u : 1u));
    fence_barrier_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(PF_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // S of tile x: columns [128x, 128x + 128); O: 256 + 128x

  bool alive = true;
  auto wait = [&](uint64_t *bar, uint32_t parity) {  // warp-uniform give-up
    if (!alive) return;
    if (!__all_sync(FULL_MASK, mbar_wait_spin(bar, parity))) {
      alive = false;
      if (lane == 0) report(a.err, PKV_DEV_ERR_TIMEOUT);
    }
  };
  if (warp == PF_SM_WARPS || warp == PF_SM_WARPS + 2) {
    // ---------------------------------------------------------- load warps
    // the first brings both tiles' Q and the K tiles, the second the V
    // tiles (on small pages a KV tile is 8 boxes per 64-dim column, and two
    // warps issue them in parallel).  A stage is refilled as soon as the
    // MMAs that read it have completed; the next tile's page ids are looked
    // up (lanes 0-7, one block each) while the warp waits.
    const uint64_t policy = l2_evict_last_policy();  // every q tile re-reads the tiles
    const int page0 = a.layer * a.num_pages;
    auto page_of = [&](int kt) -> int {  // raw page id of block lane of tile kt
      int blk = kt * 8 + (lane & 7);
      if (blk > last_blk) blk = last_blk;  // past the request: any valid block (zeroed later)
      return lane < 8 ? __ldg(a.page_table + (int64_t)b * a.max_pages + blk / a.bpp) : 0;
    };
    // pages of 128 tokens or more (a multiple of 128): a tile lies in one
    // page and comes in as NCH boxes of 128 rows
    const bool whole = (a.bpp & 7) == 0;
    auto load_kv = [&](int kt, int raw, int kv, unsigned char *dst, uint64_t *bar) {
      int blk = kt * 8 + (lane & 7);
      if (blk > last_blk) blk = last_blk;
      int pid = raw;
      if (lane < 8 && (pid < 0 || pid >= a.num_pages)) {
        if (kv == 0) report(a.err, PKV_DEV_ERR_PAGE);
        pid = 0;
      }
      const int c = pid * a.bpp + blk % a.bpp;
      const int c0 = __shfl_sync(FULL_MASK, c, 0);
      if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(NCH * 8 * PF_BLK * 128));
      __syncwarp();
      if (whole) {
        // block 0 of the tile sits at an in-page offset that is a multiple
        // of 8 blocks; one 128-row box per 64-dim column (lane ch) stays
        // inside the page
        if (lane < NCH) {
          const int pg0 = c0 / a.bpp, sub0 = c0 - pg0 * a.bpp;
          tma_load_5d(dst + lane * PF_CHUNK, &kv_map128, lane * 64, g, sub0 * PF_BLK, kv,
                      page0 + pg0, bar, policy);
        }
      } else if (lane < 8) {
        // lane i issues the boxes of block i (the issue cost is per thread)
        const int pg = c / a.bpp, sub = c - pg * a.bpp;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch)
          tma_load_5d(dst + ch * PF_CHUNK + lane * PF_BLK * 128, &kv_map, ch * 64, g,
                      sub * PF_BLK, kv, page0 + pg, bar, policy);
      }
    };
    const int kv = warp == PF_SM_WARPS ? 0 : 1;
    const int nst = kv == 0 ? S::NK : NV;
    uint64_t *full = kv == 0 ? bar_k : bar_v;
    uint64_t *freed = kv == 0 ? bar_kfree : bar_vfree;
    unsigned char *buf = kv == 0 ? ks : vs;
    int raw = page_of(0);
    if (kv == 0 && lane == 0) {
      const int ntiles = tl[1].ntok > 0 ? 2 : 1;
      mbar_arrive_expect_tx(bar_q, (uint32_t)(ntiles * NCH * a.tq * G * 128));
      for (int x = 0; x < ntiles; ++x)
        for (int ch = 0; ch < NCH; ++ch)
          tma_load_3d(qs + x * S::TILE_BYTES + ch * PF_CHUNK, &q_map, ch * 64, g * G, tl[x].t0,
                      bar_q);
    }
    for (int kt = 0; kt < nkv && alive; ++kt) {
      const int st = kt % nst, use = kt / nst;
      const int raw_next = kt + 1 < nkv ? page_of(kt + 1) : 0;
      if (use >= 1) wait(&freed[st], (uint32_t)((use - 1) & 1));
      if (!alive) break;
      load_kv(kt, raw, kv, buf + st * S::TILE_BYTES, &full[st]);
      raw = raw_next;
    }
  } else if (warp == PF_SM_WARPS + 1 || warp == PF_SM_WARPS + 3) {
    // ------------------------------------------------------------ MMA warps
    // one per tile (A: warp 9, B: warp 11), each issuing its own tile's
    // products as their inputs come: S(kt + 1) as soon as the softmax has
    // read S(kt), P.V(kt) once P(kt) is written.  The two tiles' accumulation
    // chains are independent, so the tensor pipe overlaps them.  A K or V
    // stage is free once both warps' products that read it have completed
    // (one commit per warp, also for KV tiles a shorter tile B does not read)
    const int x = warp == PF_SM_WARPS + 1 ? 0 : 1;
    const int mine = tl[x].nkv;
    constexpr uint32_t IDESC_S = bf16_idesc(PF_M, PF_N, false);
    constexpr uint32_t IDESC_O = bf16_idesc(PF_M, D, true);
    const uint64_t dq = sw128_desc(smem_addr(qs), 16, 1024);
    const uint64_t dk = sw128_desc(smem_addr(ks), 16, 1024);
    const uint64_t dv = sw128_desc(smem_addr(vs), PF_CHUNK, 1024);
    const uint64_t dp = sw128_desc(smem_addr(ps), 16, 1024);
    constexpr uint32_t TILE16 = S::TILE_BYTES >> 4;
    constexpr uint32_t P16 = S::P_BYTES >> 4;
    auto issue_s = [&](int stage) {  // S_x = Q_x K^T
      const uint64_t qb = dq + x * TILE16, kb = dk + stage * TILE16;
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = ((k >> 2) * PF_CHUNK + (k & 3) * 32) >> 4;
        tc_mma(tmem + 128 * x, qb + off, kb + off, IDESC_S, k > 0);
      }
      tc_commit(&bar_s[x]);
    };
    auto issue_o = [&](int stage, bool acc) {  // O_x += P_x V
      const uint64_t pb = dp + x * P16, vb = dv + stage * TILE16;
#pragma unroll
      for (int k = 0; k < PF_N / 16; ++k) {
        const uint32_t poff = ((k >> 2) * PF_CHUNK + (k & 3) * 32) >> 4;
        tc_mma(tmem + 256 + 128 * x, pb + poff, vb + ((k * 16 * 128) >> 4), IDESC_O,
               (acc || k > 0) ? 1u : 0u);
      }
      tc_commit(&bar_o[x]);
    };
    wait(bar_q, 0);
    wait(&bar_k[0], 0);
    if (alive && lane == 0) {
      tc_fence_after();
      if (mine > 0) issue_s(0);
      tc_commit(&bar_kfree[0]);
    }
    for (int kt = 0; kt < nkv && alive; ++kt) {
      const int nx = kt + 1;
      if (nx < nkv) {
        wait(&bar_k[nx & 1], (uint32_t)((nx >> 1) & 1));
        if (nx < mine) wait(&bar_sfree[x], (uint32_t)(kt & 1));
        if (!alive) break;
        if (lane == 0) {
          tc_fence_after();
          if (nx < mine) issue_s(nx & 1);
          tc_commit(&bar_kfree[nx & 1]);
        }
      }
      const int vst = kt % NV;
      wait(&bar_v[vst], (uint32_t)((kt / NV) & 1));
      if (!alive) break;
      tc_fence_after();
      if (kt == kt_stale && kt < mine) {
        if (x == 0) {
          // slots past the request's last position: zero the V rows, then
          // let tile B's warp (if it reads this tile) go on
          const int r0 = n - kt * PF_N;
          unsigned char *vt = vs + vst * S::TILE_BYTES;
          for (int r = r0 + lane; r < PF_N; r += 32)
            for (int c = 0; c < NCH; ++c) {
              uint4 *row = reinterpret_cast<uint4 *>(vt + c * PF_CHUNK + r * 128);
#pragma unroll
              for (int j = 0; j < 8; ++j) row[j] = make_uint4(0u, 0u, 0u, 0u);
            }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_vz);
        } else {
          wait(bar_vz, 0u);
          if (!alive) break;
        }
      }
      if (kt < mine) {
        wait(&bar_p[x], (uint32_t)(kt & 1));  // P_x[kt] written, O_x rescaled
        if (!alive) break;
        if (lane == 0) {
          tc_fence_after();
          issue_o(vst, kt > 0);
        }
      }
      if (lane == 0) tc_commit(&bar_vfree[vst]);
    }
    // drain: every MMA of both warps has completed
    if (lane == 0) {
      tc_commit(bar_fin);
      if (!mbar_wait_spin(bar_fin, 0)) report(a.err, PKV_DEV_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp < PF_SM_WARPS) {
    // ------------------------------------------------------ softmax warps
    // warpgroup x owns tile x; thread r of the group owns row r (TMEM lane)
    const int x = warp >> 2;
    const PfTile T = x ? tl[1] : tl[0];
    const int r = tid & 127;
    const int tok = r / G;
    const int hj = r % G;
    const bool valid = tok < T.ntok && r < a.tq * G && T.t0 + tok < a.T;
    const int p = T.pos0 + tok;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tm_s = tmem + 128 * x, tm_o = tmem + 256 + 128 * x;
    unsigned char *pbuf = ps + x * S::P_BYTES;
    // l_run: sum of the fp32 weights (for lse); w_run: sum of the weights as
    // rounded to bf16 for P.V (normalises O, so the output is a weighted
    // mean of the values with the weights the tensor cores actually used)
    float m_run = -INFINITY, l_run = 0.0f, w_run = 0.0f;
    for (int kt = 0; kt < T.nkv; ++kt) {
      if (!__all_sync(FULL_MASK, mbar_wait_spin(&bar_s[x], (uint32_t)(kt & 1)))) {  // warp-uniform
        alive = false;
        if (lane == 0) report(a.err, PKV_DEV_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tm_s + lane_off + c * 32, sr[c]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar_sfree[x]);  // the tensor cores may overwrite S now
      // causal mask (raw scores; only tiles that reach past some row's
      // position need it)
      const int lim = valid ? p - kt * PF_N : -1;  // keys <= lim are allowed
      float mx = -INFINITY;
      if (__any_sync(FULL_MASK, lim < PF_N - 1)) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float v = (c * 32 + j <= lim) ? __uint_as_float(sr[c][j]) : -INFINITY;
            sr[c][j] = __float_as_uint(v);
            mx = fmaxf(mx, v);
          }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(sr[c][j]));
      }
      mx *= a.qscale;  // log2 units (qscale > 0)
      float m_ref = m_run, alpha = 1.0f;
      if (mx > m_run + PF_TAU) {
        m_ref = mx;
        alpha = fast_exp2(m_run - mx);  // 0 when m_run = -inf
      }
      const float m_use = m_ref == -INFINITY ? 0.0f : m_ref;
      // p = 2^(s * qscale - m), two at a time
      const f32x2 sc2 = pack2(a.qscale, a.qscale), nm2 = pack2(-m_use, -m_use);
      f32x2 acc = pack2(0.0f, 0.0f), wacc = pack2(0.0f, 0.0f);
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float2 t = unpack2(
              ffma2(pack2(__uint_as_float(sr[c][j]), __uint_as_float(sr[c][j + 1])), sc2, nm2));
          const float p0 = fast_exp2(t.x), p1 = fast_exp2(t.y);
          const f32x2 pp = pack2(p0, p1);
          acc = fadd2(acc, pp);
          const uint32_t w = pack_bf16x2(p0, p1);
          wacc = fadd2(wacc, pack2(bf16lo(w), bf16hi(w)));
          pk[(c * 32 + j) >> 1] = w;
        }
      const float2 accf = unpack2(acc), waccf = unpack2(wacc);
      l_run = l_run * alpha + (accf.x + accf.y);
      w_run = w_run * alpha + (waccf.x + waccf.y);
      const bool resc = kt > 0 && alpha != 1.0f;
      m_run = m_ref;
      if (kt > 0) {
        // P.V[kt-1] done: O is stable and the P buffer free
        if (!__all_sync(FULL_MASK, mbar_wait_spin(&bar_o[x], (uint32_t)((kt - 1) & 1)))) {
          alive = false;
          if (lane == 0) report(a.err, PKV_DEV_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        if (__any_sync(FULL_MASK, resc)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tm_o + lane_off + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(tm_o + lane_off + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      // P row r, keys 0..127, as two 64-key swizzle columns (the A operand
      // of P.V, K-major)
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint4 *dst =
              reinterpret_cast<uint4 *>(pbuf + c * PF_CHUNK + r * 128 + ((j ^ (r & 7)) << 4));
          *dst = make_uint4(pk[c * 32 + 4 * j], pk[c * 32 + 4 * j + 1], pk[c * 32 + 4 * j + 2],
                            pk[c * 32 + 4 * j + 3]);
        }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_p[x]);
    }
    if (T.nkv > 0) {
      if (alive && __all_sync(FULL_MASK, mbar_wait_spin(&bar_o[x], (uint32_t)((T.nkv - 1) & 1)))) {
        tc_fence_after();
        const float inv = w_run > 0.0f ? 1.0f / w_run : 0.0f;
        const int t = T.t0 + tok;
        uint16_t *orow = a.out + ((int64_t)t * Hq + g * G + hj) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tm_o + lane_off + c * 32, o);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv);
              *reinterpret_cast<uint4 *>(orow + c * 32 + j) = w;
            }
          }
        }
        if (valid && a.lse != nullptr)
          a.lse[(int64_t)t * Hq + g * G + hj] =
              l_run > 0.0f ? (m_run + __log2f(l_run)) * 0.69314718055994530942f : -INFINITY;
      } else if (lane == 0) {
        report(a.err, PKV_DEV_ERR_TIMEOUT);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(PF_TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 pf_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// (head_dim, kv head, slot, K/V, layer * num_pages + page); one box = 64
// dims x 16 slots of one kv head, K or V, 128-byte swizzled
static int encode_kv_map(CUtensorMap *map, const void *cache, const pkv_cache_t *g,
                         int box_rows) {
  auto enc = pf_encoder();
  if (enc == nullptr) return PKV_ERR_CUDA;
  const cuuint64_t D = (cuuint64_t)g->head_dim, H = (cuuint64_t)g->num_kv_heads;
  const cuuint64_t PS = (cuuint64_t)g->page_size;
  const cuuint64_t dims[5] = {D, H, PS, 2, (cuuint64_t)g->num_layers * (cuuint64_t)g->num_pages};
  const cuuint64_t strides[4] = {D * 2, H * D * 2, PS * H * D * 2, 2 * PS * H * D * 2};
  const cuuint32_t box[5] = {64, 1, (cuuint32_t)box_rows, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(cache), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_UNSUPPORTED;
}

// q [T][Hq][D]: one box = 64 dims x G heads x tq tokens, 128-byte swizzled
static int encode_q_map(CUtensorMap *map, const void *q, int T, int Hq, int D, int G, int tq) {
  auto enc = pf_encoder();
  if (enc == nullptr) return PKV_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)tq};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_UNSUPPORTED;
}

struct PfWs {
  size_t tile_start, order, hdr, total;
};
static PfWs pf_ws(int batch) {
  PfWs w;
  w.tile_start = 0;
  w.order = align_up((size_t)(batch + 1) * sizeof(int32_t), 256);
  w.hdr = w.order + align_up((size_t)batch * sizeof(int32_t), 256);
  w.total = w.hdr + 256;
  return w;
}

template <int D>
static int launch_prefill(const PfArgs &a, const CUtensorMap &kvm, const CUtensorMap &kvm128,
                          const CUtensorMap &qm, int max_units, cudaStream_t st) {
  using S = PfShape<D>;
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(prefill_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::SMEM_BYTES) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev] = true;
  }
  if (launch_pdl(prefill_plan_kernel, dim3(1), dim3(PF_PLAN_THREADS), 0, st, a) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (launch_pdl(prefill_attn_kernel<D>, dim3((unsigned)max_units), dim3(PF_THREADS),
                 (size_t)S::SMEM_BYTES, st, a, kvm, kvm128, qm) != cudaSuccess)
    return PKV_ERR_CUDA;
  return launch_status();
}

}  // namespace pkv

extern "C" size_t pkv_prefill_workspace_bytes(int batch) {
  if (batch <= 0) return 0;
  return pkv::pf_ws(batch).total;
}

extern "C" int pkv_prefill_attn(const pkv_cache_t *geom, const void *cache, int layer,
                                const void *q, int num_qo_heads, float sm_scale, int total_tokens,
                                const int32_t *qo_indptr, const int32_t *page_table,
                                int max_pages, const int32_t *seq_lens, const int32_t *active,
                                int batch, void *out, float *lse, void *workspace,
                                size_t workspace_bytes, int32_t *err_word, void *stream) {
  using namespace pkv;
  int st = check_geometry(geom);
  if (st != PKV_OK) return st;
  if (!cache || !q || !qo_indptr || !page_table || !seq_lens || !active || !out)
    return PKV_ERR_INVALID_ARG;
  if (batch <= 0 || total_tokens <= 0 || max_pages <= 0 || layer < 0 ||
      layer >= geom->num_layers || num_qo_heads <= 0 || num_qo_heads % geom->num_kv_heads != 0)
    return PKV_ERR_INVALID_ARG;
  if (!(sm_scale > 0.0f)) return PKV_ERR_INVALID_ARG;  // the row maximum is taken on raw scores
  const int D = geom->head_dim;
  const int G = num_qo_heads / geom->num_kv_heads;
  if ((D != 64 && D != 128) || geom->page_size % PF_BLK != 0 || geom->page_size > 1024 ||
      G > PF_M)
    return PKV_ERR_UNSUPPORTED;
  const int64_t max_tokens = (int64_t)max_pages * geom->page_size;
  if (max_tokens > INT32_MAX || (int64_t)geom->num_layers * geom->num_pages > INT32_MAX)
    return PKV_ERR_UNSUPPORTED;
  if (!aligned16(cache) || !aligned16(q) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
  const PfWs wl = pf_ws(batch);
  if (workspace == nullptr || workspace_bytes < wl.total) return PKV_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return PKV_ERR_INVALID_ARG;

  PfArgs a;
  a.layer = layer;
  a.num_pages = geom->num_pages;
  a.bpp = geom->page_size / PF_BLK;
  a.num_kv_heads = geom->num_kv_heads;
  a.num_qo_heads = num_qo_heads;
  a.group = G;
  a.tq = PF_M / G;
  a.T = total_tokens;
  a.qscale = sm_scale * 1.44269504088896340736f;
  a.qo_indptr = qo_indptr;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.max_tokens = max_tokens;
  a.seq_lens = seq_lens;
  a.active = active;
  a.batch = batch;
  a.out = static_cast<uint16_t *>(out);
  a.lse = lse;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  a.tile_start = reinterpret_cast<int32_t *>(ws + wl.tile_start);
  a.order = reinterpret_cast<int32_t *>(ws + wl.order);
  a.hdr = reinterpret_cast<PfHeader *>(ws + wl.hdr);
  a.err = err_word;
  // units: sum over requests of ceil(nt_b / 2), nt_b = ceil(q_b / tq), with
  // sum nt_b <= ceil(T / tq) + B, so at most (ceil(T / tq) + 2B + 1) / 2
  // (a CTA past the planner's count exits at once, but holds an SM while
  // it does)
  const int64_t tiles_bound = (int64_t)(total_tokens + a.tq - 1) / a.tq + batch;
  const int64_t max_units = ((tiles_bound + batch + 1) / 2) * geom->num_kv_heads;
  if (max_units > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  alignas(64) CUtensorMap kvm, kvm128, qm;
  st = encode_kv_map(&kvm, cache, geom, PF_BLK);
  if (st != PKV_OK) return st;
  // 128-row boxes (used only when a page holds a multiple of 128 tokens)
  st = encode_kv_map(&kvm128, cache, geom, geom->page_size % PF_N == 0 ? PF_N : PF_BLK);
  if (st != PKV_OK) return st;
  st = encode_q_map(&qm, q, total_tokens, num_qo_heads, D, G, a.tq);
  if (st != PKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return D == 128 ? launch_prefill<128>(a, kvm, kvm128, qm, (int)max_units, s)
                  : launch_prefill<64>(a, kvm, kvm128, qm, (int)max_units, s);
}
