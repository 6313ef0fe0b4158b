// decode_attn.cu -- grouped-query decode attention over the paged cache:
// attn_wrapper.run(q, kv_cache) of "Adding a Model" (vox-serve docs),
// section "1. The model code", for the layout
// [num_layers, num_pages, 2, page_size, num_kv_heads, head_dim].
//
// Design (HBM-bound; CUDA cores, no tensor cores):
//  * blocks: the kernel streams a row's context in 16-token blocks; a page
//    of page_size tokens (any multiple of 16) is page_size / 16 blocks.
//  * work units: a row's blocks are cut into fixed 32-block (512-token)
//    splits; a unit is one (row, split, kv head, q-head block).  The split size does
//    not depend on the batch, so a row's result depends on its inputs only.
//  * a one-CTA planner lists the splits of the active rows and resets the
//    scheduling counter, so the launch shapes stay static.  Units are handed
//    out largest first: every full 32-block split (prefix sums over the
//    rows), then each row's shorter last split in descending size (a
//    counting sort).  The order only decides which CTA takes a unit, never
//    how a row's result is formed.  The planner reads only lengths and
//    flags, which no kernel of this library writes, so it does its work
//    while its predecessor (the KV append) still runs and waits for that
//    predecessor only at its end.
//  * a persistent grid (SMs x resident CTAs): CTA i starts on unit i and
//    pulls the rest from an atomic counter.  Each of a CTA's 4 warps streams its blocks of the unit
//    (round-robin) through its own ring of NS shared-memory stages; a stage
//    is one block of one kv head -- 16 K rows + 16 V rows, each head_dim bf16
//    contiguous in HBM -- brought in by one tiled tensor TMA
//    (cp.async.bulk.tensor) completing on the stage's mbarrier.  The ring runs on
//    into the next unit, so its pages are in flight while the current unit
//    is merged.  Waits are bounded.
//  * GQA sharing: a warp holds the q of all the group's heads in registers,
//    so every K / V element is read from shared memory and converted once
//    and used for every head of the group.
//  * lanes: 8 lanes share a token, each lane owns head_dim/8 dims read as
//    16-byte vectors (conflict-free); q.k partial sums are summed over the 8
//    lanes with 3 xor-shuffles; the online softmax runs in the log2 domain
//    with a lazy maximum (rescale only when a score beats the running
//    maximum by more than 8).
//  * a page's two 8-token batches are processed together (more independent
//    work per warp between the shuffle steps).
//  * per unit, the 4 lane groups of a warp merge with shuffles and the 4
//    warps through shared memory into one (m, l, o) partial; a merge kernel
//    then folds each row's partials in split order and writes the zeros of
//    padding rows.  No fences, tickets or
//    blocking atomics sit in the streaming loop: the next unit's id is
//    fetched one unit ahead.
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <utility>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int ATTN_WARPS = 4;
constexpr int ATTN_THREADS = ATTN_WARPS * 32;
constexpr int ATTN_PAGES_PER_SPLIT = 32;  // 16-token blocks per split
constexpr int ATTN_PAGE = 16;             // tokens per block (a page is page_size / 16 blocks)
constexpr int ATTN_MAX_PAGE_SIZE = 1024;
constexpr float ATTN_TAU = 8.0f;       // lazy-rescale threshold (log2 units)
constexpr float ATTN_NEG = -1.0e30f;   // "no score yet" (finite: keeps 2^(s-m) at 0)
constexpr float LN2 = 0.69314718055994530942f;
constexpr float LOG2E = 1.44269504088896340736f;
constexpr int PLAN_THREADS = 1024;

struct PlanHeader {
  int32_t counter;      // next unit to hand out
  int32_t total_units;
  int32_t total_splits;
  int32_t full_splits;  // splits of 32 whole blocks; they come first
};

struct AttnArgs {
  const unsigned char *cache;  // byte address of the cache
  int64_t layer_off;           // bytes
  int64_t page_stride;         // bytes
  int64_t kv_stride;           // bytes
  int64_t tok_stride;          // bytes
  int num_pages;
  int num_kv_heads;
  int head_dim;
  int layer;
  const uint16_t *q;           // [B][Hq][D] bf16 bits
  int num_qo_heads;
  int group;                   // Hq / Hkv
  int qblocks;                 // q-head blocks per kv head
  int gp;                      // q heads per block
  float qscale;                // sm_scale * log2(e)
  const int32_t *page_table;
  int max_pages;
  int bpp;                     // 16-token blocks per page
  int64_t max_tokens;          // max_pages * page_size
  const int32_t *seq_lens;
  const int32_t *active;
  int batch;
  void *out;
  int out_fp32;
  float *lse;
  float *ws_o;                 // [B][Hq][nsplit_max][D]
  float2 *ws_ml;               // [B][Hq][nsplit_max]
  int32_t *row_start;          // [B + 1] first full split of each row, then
                               // [B] rows of the short last splits, longest first
  int32_t *part_rows;          // row_start + B + 1
  PlanHeader *plan;
  int nsplit_max;
  int32_t *err;
};

__device__ __forceinline__ void store_out(const AttnArgs &a, int64_t idx, float v) {
  if (a.out_fp32)
    static_cast<float *>(a.out)[idx] = v;
  else
    static_cast<uint16_t *>(a.out)[idx] = (uint16_t)f32_to_bf16_bits(v);
}

// 16-token blocks of row b (0 for padding and rejected rows)
__device__ __forceinline__ int row_blocks(const AttnArgs &a, int b, bool *bad) {
  *bad = false;
  if (!a.active[b]) return 0;
  const int n = a.seq_lens[b];
  if (n < 1 || (int64_t)n > a.max_tokens) {
    *bad = true;
    return 0;
  }
  return (n + ATTN_PAGE - 1) / ATTN_PAGE;
}

// ---------------------------------------------------------------------------
// planner: one CTA
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(PLAN_THREADS) attn_plan_kernel(const AttnArgs a) {
  constexpr int SPL = ATTN_PAGES_PER_SPLIT;
  __shared__ int32_t scan[PLAN_THREADS];
  __shared__ int32_t carry;
  __shared__ int32_t bin[SPL];  // short last splits per size, then the next slot of each size
  // No early launch of dependents: a kernel after this one starts only once
  // the plan is complete, so it may read the plan before its own wait.
  const int tid = threadIdx.x;
  const int HB = a.num_kv_heads * a.qblocks;
  if (tid == 0) carry = 0;
  if (tid < SPL) bin[tid] = 0;
  __syncthreads();
  for (int base = 0; base < a.batch; base += PLAN_THREADS) {
    const int b = base + tid;
    int nf = 0;
    if (b < a.batch) {
      bool bad;
      const int nb = row_blocks(a, b, &bad);
      if (bad) report(a.err, PKV_DEV_ERR_SEQ_LEN);
      nf = nb / SPL;
      if (nb % SPL) atomicAdd(&bin[nb % SPL], 1);
    }
    // inclusive scan of the full splits over the block (Hillis-Steele)
    scan[tid] = nf;
    __syncthreads();
    for (int off = 1; off < PLAN_THREADS; off <<= 1) {
      const int v = tid >= off ? scan[tid - off] : 0;
      __syncthreads();
      scan[tid] += v;
      __syncthreads();
    }
    if (b < a.batch) a.row_start[b] = carry + scan[tid] - nf;
    __syncthreads();
    if (tid == PLAN_THREADS - 1) carry += scan[tid];
    __syncthreads();
  }
  // first slot of each size, longest first: bin[r] = rows with a longer
  // short split
  if (tid == 0) {
    int acc = 0;
    for (int r = SPL - 1; r >= 1; --r) {
      const int c = bin[r];
      bin[r] = acc;
      acc += c;
    }
    a.row_start[a.batch] = carry;
    a.plan->counter = 0;
    a.plan->full_splits = carry;
    a.plan->total_splits = carry + acc;
    a.plan->total_units = (carry + acc) * HB;
  }
  __syncthreads();
  // the rows of the short splits in their slots (the order within a size
  // does not matter: each unit writes its own partial)
  for (int b = tid; b < a.batch; b += PLAN_THREADS) {
    bool bad;
    const int r = row_blocks(a, b, &bad) % SPL;
    if (r) a.part_rows[atomicAdd(&bin[r], 1)] = b;
  }
  // completes only after the predecessor has: the persistent kernel, which
  // waits for this grid, then sees the predecessor's cache writes too
  pdl_wait();
}

// ---------------------------------------------------------------------------
// the persistent attention kernel
// ---------------------------------------------------------------------------
template <int D, int GP, int NS>
struct AttnShape {
  static constexpr int T = 8 / GP;              // tokens per lane group per batch
  static constexpr int TOK_PER_BATCH = 4 * T;   // tokens per warp per batch
  static constexpr int NB = ATTN_PAGE / TOK_PER_BATCH;  // batches per page
  static constexpr int DPL = D / 8;             // dims per lane
  static constexpr int NCH = DPL / 8;           // 16-byte chunks per lane per row
  static constexpr int NP = DPL / 2;            // fp32 pairs per lane per row
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int STAGE_BYTES = 2 * ATTN_PAGE * ROW_BYTES;
  static constexpr int RING_BYTES = ATTN_WARPS * NS * STAGE_BYTES;
  static constexpr int QBUF_BYTES = 2 * GP * D * 2;         // staged q of cur / next (bf16)
  static constexpr int RED_O_BYTES = ATTN_WARPS * GP * D * 4;
  static constexpr int RED_ML_BYTES = ATTN_WARPS * GP * 8;
  static constexpr int BAR_BYTES = ATTN_WARPS * NS * 8 + 2 * 8;
  static constexpr int SMEM_BYTES =
      RING_BYTES + QBUF_BYTES + RED_O_BYTES + RED_ML_BYTES + BAR_BYTES + 128;
  static_assert(GP == 2 || GP == 4 || GP == 8, "GP");
  static_assert(D == 64 || D == 128, "D");
};

struct Unit {
  int valid;
  int b, split, g, h0, nh;
  int n, p_begin, p_count;
  int bad;  // the row's length disagrees with the plan: skipped, reported
};

constexpr int ATTN_SMEM_ROWS = 512;  // rows whose split table lives in shared memory
// static shared memory of the persistent kernel (unit ring + split table)
constexpr int ATTN_STATIC_SMEM = 4 * (4 + 1 + (2 * ATTN_SMEM_ROWS + 1) + ATTN_SMEM_ROWS) + 128;
constexpr int SM_SMEM_BYTES = 228 * 1024;  // shared memory of one SM (1 KB reserved per CTA)

// rs: first full split of each row [B + 1], followed by the rows of the
// short splits; seq: lengths [B] (each in shared or global memory).  Units
// [0, full * HB) are full splits, the rest the short last splits in the
// planner's order.
__device__ __forceinline__ Unit decode_unit(const AttnArgs &a, int u, int gp, int total_units,
                                            int full, const int32_t *rs, const int32_t *seq) {
  Unit U;
  const int HB = a.num_kv_heads * a.qblocks;
  U.valid = u < total_units;
  U.b = U.split = U.g = U.h0 = U.nh = U.n = U.p_begin = U.p_count = U.bad = 0;
  if (!U.valid) return U;
  const int su = u / HB, hb = u % HB;
  if (su < full) {
    // row of full split `su`: the last b with rs[b] <= su (a row without
    // full splits shares its rs with the next row, so it is never chosen)
    int lo = 0, hi = a.batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (rs[mid] <= su)
        lo = mid;
      else
        hi = mid - 1;
    }
    U.b = lo;
    U.split = su - rs[lo];
  } else {
    U.b = rs[a.batch + 1 + su - full];
    U.split = -1;  // the row's last split, set below
  }
  U.g = hb / a.qblocks;
  const int qb = hb % a.qblocks;
  U.h0 = U.g * a.group + qb * gp;
  U.nh = min(gp, a.group - qb * gp);
  U.n = seq[U.b];
  const bool n_ok = U.n >= 1 && (int64_t)U.n <= a.max_tokens;
  const int npages = n_ok ? (U.n + ATTN_PAGE - 1) / ATTN_PAGE : 0;
  if (U.split < 0) U.split = npages / ATTN_PAGES_PER_SPLIT;
  U.p_begin = U.split * ATTN_PAGES_PER_SPLIT;
  U.p_count = min(npages - U.p_begin, ATTN_PAGES_PER_SPLIT);
  U.bad = 0;
  if (U.p_count <= 0 || U.split >= a.nsplit_max) {
    // the row's length no longer matches the plan the unit came from (it
    // changed after pkv_decode_plan): no blocks are read and no partial is
    // written for it
    U.bad = 1;
    U.p_count = 0;
    report(a.err, PKV_DEV_ERR_SEQ_LEN);
  }
  return U;
}

__device__ __forceinline__ int warp_pages(const Unit &U, int warp) {
  if (!U.valid || U.p_count <= warp) return 0;
  return (U.p_count - warp + ATTN_WARPS - 1) / ATTN_WARPS;
}

// barrier 1 over the CTA's 128 threads (barrier 0 stays __syncthreads)
__device__ __forceinline__ void named_barrier_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(ATTN_THREADS) : "memory");
}

template <int D, int GP, int NS>
__global__ void __launch_bounds__(ATTN_THREADS, 2)
    attn_persistent_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmap) {
  using S = AttnShape<D, GP, NS>;
  constexpr int T = S::T, NCH = S::NCH, NP = S::NP, NB = S::NB;
  static_assert(2 * (S::SMEM_BYTES + ATTN_STATIC_SMEM + 1024) <= SM_SMEM_BYTES,
                "two CTAs per SM");

  extern __shared__ __align__(128) unsigned char smem_raw[];
  // stage buffers start on a 128-byte boundary
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  unsigned char *p = smem + S::RING_BYTES;
  uint16_t *qbuf = reinterpret_cast<uint16_t *>(p);  // [2][GP][D]
  p += S::QBUF_BYTES;
  float *red_o = reinterpret_cast<float *>(p);  // [4][GP][D]
  p += S::RED_O_BYTES;
  float2 *red_ml = reinterpret_cast<float2 *>(p);  // [4][GP]
  p += S::RED_ML_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(p);
  uint64_t *qbars = bars + ATTN_WARPS * NS;  // [2]
  __shared__ int32_t s_unit[4];  // unit ids, circular: ordinal k at [k & 3]
  __shared__ int32_t s_rs[2 * ATTN_SMEM_ROWS + 1];
  __shared__ int32_t s_seq[ATTN_SMEM_ROWS];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int grp = lane >> 3;
  const int li = lane & 7;
  const int gbase = lane & 24;  // first lane of the lane group
  const int h_own = li / T;     // after the reduce-scatter, lane li holds value
  const int tt_own = li % T;    // li = (head h_own, token tt_own) of its group
  const int Hq = a.num_qo_heads;

  unsigned char *ring = smem + warp * NS * S::STAGE_BYTES;
  uint64_t *wbars = bars + warp * NS;
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&wbars[s], 1);
    if (warp == 0) {
      mbar_init(&qbars[0], 1);
      mbar_init(&qbars[1], 1);
    }
    fence_barrier_init();
  }
  // The plan, the lengths and flags and the page table were final before
  // this grid's predecessor started: the planner lets no kernel start before
  // it completes, and the library's other kernels wait for their own
  // predecessor before they let a dependent start.  So the split table is
  // read, the first unit (unit blockIdx.x) decoded and its page ids loaded
  // while the predecessor (the KV append) may still run; q, the cache and
  // the unit counter are read only after the wait.
  const bool small_batch = a.batch <= ATTN_SMEM_ROWS;
  __shared__ int32_t s_full;  // full splits (read once per unit, not held in registers)
  const int total_units = a.plan->total_units;
  const int nshort = a.plan->total_splits - a.plan->full_splits;
  if (tid == 0) s_full = a.plan->full_splits;
  if (small_batch) {
    for (int i = tid; i <= a.batch + nshort; i += ATTN_THREADS) s_rs[i] = a.row_start[i];
    for (int b = tid; b < a.batch; b += ATTN_THREADS) s_seq[b] = a.seq_lens[b];
  }
  __syncthreads();
  const int32_t *rs = small_batch ? s_rs : a.row_start;
  const int32_t *seq = small_batch ? s_seq : a.seq_lens;
  const uint64_t policy = l2_evict_first_policy();
  const int layer_page0 = a.layer * a.num_pages;

  // the warp's blocks of a unit: lane i holds the i-th as page * bpp + the
  // block's index inside its page
  auto load_pids = [&](const Unit &U, int cnt) -> int {
    int pid = 0;
    if (lane < cnt) {
      const int blk = U.p_begin + warp + lane * ATTN_WARPS;
      const int pg = a.bpp == 1 ? blk : blk / a.bpp;
      // the unit's blocks lie inside the row's page-table row (decode_unit
      // checked the length); the clamp keeps the read there regardless
      pid = __ldg(a.page_table + (int64_t)U.b * a.max_pages + min(pg, a.max_pages - 1));
      if (pid < 0 || pid >= a.num_pages) {
        report(a.err, PKV_DEV_ERR_PAGE);
        pid = 0;
      }
      pid = pid * a.bpp + (blk - pg * a.bpp);
    }
    return pid;
  };
  int ordinal = 0;
  // every CTA starts on unit blockIdx.x; later units come from the counter
  // (offset by the grid), so a batch with fewer units than CTAs gives each
  // CTA at most one instead of two to the first half of the grid
  Unit cur = decode_unit(a, (int)blockIdx.x, GP, total_units, s_full, rs, seq);
  int cur_cnt = warp_pages(cur, warp);
  int pid_cur = load_pids(cur, cur_cnt);

  pdl_wait();     // the predecessor: the cache (the append), q, the unit counter
  pdl_trigger();  // the merge kernel may queue behind this grid now
  if (tid == 0) {
    s_unit[0] = (int)blockIdx.x;
    s_unit[1] = (int)gridDim.x + atomicAdd(&a.plan->counter, 1);
  }
  __syncthreads();
  Unit nxt = decode_unit(a, s_unit[1], GP, total_units, s_full, rs, seq);
  int nxt_cnt = warp_pages(nxt, warp);
  int next_id = 0;  // id of the unit after next, fetched a unit ahead (thread 0)
  int pid_nxt = load_pids(nxt, nxt_cnt);

  // q rows of a unit's heads (contiguous in HBM) into q buffer `buf`
  auto stage_q = [&](const Unit &U, int buf) {
    if (tid == 0 && U.valid) {
      fence_proxy_async_smem();
      const uint32_t bytes = (uint32_t)(U.nh * D * 2);
      mbar_arrive_expect_tx(&qbars[buf], bytes);
      bulk_copy_g2s(qbuf + buf * GP * D, a.q + ((int64_t)U.b * Hq + U.h0) * D, bytes, &qbars[buf]);
    }
  };
  stage_q(cur, 0);
  stage_q(nxt, 1);

  // ring positions
  int iss_slot = 0, con_slot = 0;
  uint32_t con_phase = 0;
  int inflight = 0;
  // issue pointer: which of (cur, nxt) and which of the warp's pages of it
  int iss_u = 0, iss_i = 0;
  bool dead = false;  // a bounded wait gave up: stop streaming, keep the barriers

  // one tensor TMA brings the block's 16 K rows and 16 V rows of kv head g
  auto issue_one = [&](int g, int pids, int i) {
    const int c = __shfl_sync(FULL_MASK, pids, i);
    if (lane == 0) {
      const int pid = a.bpp == 1 ? c : c / a.bpp;
      const int sub = c - pid * a.bpp;
      uint64_t *bar = &wbars[iss_slot];
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, S::STAGE_BYTES);
      tma_load_5d(ring + iss_slot * S::STAGE_BYTES, &tmap, 0, g, sub * ATTN_PAGE, 0,
                  layer_page0 + pid, bar, policy);
    }
    iss_slot = iss_slot + 1 == NS ? 0 : iss_slot + 1;
    ++inflight;
  };
  auto top_up = [&]() {
    if (dead) return;
    while (inflight < NS) {
      if (iss_u == 0) {
        if (iss_i < cur_cnt) {
          issue_one(cur.g, pid_cur, iss_i++);
          continue;
        }
        iss_u = 1;
        iss_i = 0;
      }
      if (iss_i < nxt_cnt) {
        issue_one(nxt.g, pid_nxt, iss_i++);
        continue;
      }
      break;
    }
  };

  f32x2 q2[GP][NP];
  f32x2 o2[GP][NP];
  float m_all[GP];  // running maximum per head (log2 units), shared by the lane group
  float m_own, l_own;

  while (cur.valid) {
    if (tid == 0) next_id = (int)gridDim.x + atomicAdd(&a.plan->counter, 1);  // used at the epilogue
    top_up();
    // q of the lane's dims for every head of the block, pre-scaled to log2 units
    const int qb_idx = ordinal & 1;
    if (!mbar_wait(&qbars[qb_idx], (uint32_t)((ordinal >> 1) & 1)) && lane == 0)
      report(a.err, PKV_DEV_ERR_TIMEOUT);
    const uint16_t *qsrc = qbuf + qb_idx * GP * D;
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      m_all[h] = ATTN_NEG;
#pragma unroll
      for (int j = 0; j < NP; ++j) o2[h][j] = 0ull;
      if (h < cur.nh) {
        const uint4 *qr = reinterpret_cast<const uint4 *>(qsrc + h * D);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          float f[8];
          unpack8(qr[li + 8 * c], f);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            q2[h][4 * c + e] = pack2(f[2 * e] * a.qscale, f[2 * e + 1] * a.qscale);
        }
      } else {
#pragma unroll
        for (int j = 0; j < NP; ++j) q2[h][j] = 0ull;
      }
    }
    m_own = ATTN_NEG;
    l_own = 0.0f;
    const int n = cur.n;
    const int tok_base = cur.p_begin * ATTN_PAGE;

    for (int i = 0; i < cur_cnt && !dead; ++i) {
      const bool landed = mbar_wait(&wbars[con_slot], con_phase);
      if (!__all_sync(FULL_MASK, landed)) {  // warp-uniform give-up
        dead = true;
        if (lane == 0) report(a.err, PKV_DEV_ERR_TIMEOUT);
        break;
      }
      const unsigned char *kst = ring + con_slot * S::STAGE_BYTES;
      const unsigned char *vst = kst + ATTN_PAGE * S::ROW_BYTES;
      const int tok0 = tok_base + (warp + i * ATTN_WARPS) * ATTN_PAGE;
      const bool ragged = tok0 + ATTN_PAGE > n;

      // ---- q.k for every batch of the page: x[b][h * T + tt] ----------
      float x[NB][8];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
#pragma unroll
        for (int tt = 0; tt < T; ++tt) {
          const int tok = b * S::TOK_PER_BATCH + grp * T + tt;
          const uint4 *kr = reinterpret_cast<const uint4 *>(kst + tok * S::ROW_BYTES);
          f32x2 k2[NP];
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            const uint4 w = kr[li + 8 * c];
            k2[4 * c + 0] = bf16x2_to_f32x2(w.x);
            k2[4 * c + 1] = bf16x2_to_f32x2(w.y);
            k2[4 * c + 2] = bf16x2_to_f32x2(w.z);
            k2[4 * c + 3] = bf16x2_to_f32x2(w.w);
          }
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            f32x2 acc = fmul2(q2[h][0], k2[0]);
#pragma unroll
            for (int j = 1; j < NP; ++j) acc = ffma2(q2[h][j], k2[j], acc);
            const float2 r = unpack2(acc);
            x[b][h * T + tt] = r.x + r.y;
          }
        }
      }
      // ---- reduce-scatter over the 8 lanes of a group: lane li ends with
      //      the full dot product of value li, for each batch ------------
      float s[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float y[4], z[2];
        const bool u4 = li & 4, u2 = li & 2, u1 = li & 1;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float send = u4 ? x[b][k] : x[b][k + 4];
          const float keep = u4 ? x[b][k + 4] : x[b][k];
          y[k] = keep + __shfl_xor_sync(FULL_MASK, send, 4);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float send = u2 ? y[k] : y[k + 2];
          const float keep = u2 ? y[k + 2] : y[k];
          z[k] = keep + __shfl_xor_sync(FULL_MASK, send, 2);
        }
        const float send = u1 ? z[0] : z[1];
        const float keep = u1 ? z[1] : z[0];
        s[b] = keep + __shfl_xor_sync(FULL_MASK, send, 1);
        if (ragged && tok0 + b * S::TOK_PER_BATCH + grp * T + tt_own >= n) s[b] = -INFINITY;
      }
      // ---- online softmax with a lazy maximum -------------------------
      bool need = false;
#pragma unroll
      for (int b = 0; b < NB; ++b) need |= s[b] > m_own + ATTN_TAU;
      if (__any_sync(FULL_MASK, need)) {
        float bm = s[0];  // maximum of the page for head h_own
#pragma unroll
        for (int b = 1; b < NB; ++b) bm = fmaxf(bm, s[b]);
#pragma unroll
        for (int off = 1; off < T; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, off));
        float m_own_new = m_own;
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          const float mh = __shfl_sync(FULL_MASK, bm, gbase | (h * T));
          const float mn = fmaxf(m_all[h], mh);
          const float sc = fast_exp2(m_all[h] - mn);
          const f32x2 sc2 = pack2(sc, sc);
#pragma unroll
          for (int j = 0; j < NP; ++j) o2[h][j] = fmul2(o2[h][j], sc2);
          m_all[h] = mn;
          if (h == h_own) m_own_new = mn;
        }
        l_own *= fast_exp2(m_own - m_own_new);
        m_own = m_own_new;
      }
      // ---- probabilities, gathered to every lane of the group ----------
      float pv[NB][8];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float pr = fast_exp2(s[b] - m_own);
        l_own += pr;
#pragma unroll
        for (int v = 0; v < 8; ++v) pv[b][v] = __shfl_sync(FULL_MASK, pr, gbase | v);
      }
      // ---- p.v -------------------------------------------------------
#pragma unroll
      for (int b = 0; b < NB; ++b) {
#pragma unroll
        for (int tt = 0; tt < T; ++tt) {
          const int tok = b * S::TOK_PER_BATCH + grp * T + tt;
          const uint4 *vr = reinterpret_cast<const uint4 *>(vst + tok * S::ROW_BYTES);
          f32x2 v2[NP];
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            const uint4 w = vr[li + 8 * c];
            v2[4 * c + 0] = bf16x2_to_f32x2(w.x);
            v2[4 * c + 1] = bf16x2_to_f32x2(w.y);
            v2[4 * c + 2] = bf16x2_to_f32x2(w.z);
            v2[4 * c + 3] = bf16x2_to_f32x2(w.w);
          }
          if (ragged && tok0 + tok >= n) {
            // rows past the end of the sequence may hold any bits
#pragma unroll
            for (int j = 0; j < NP; ++j) v2[j] = 0ull;
          }
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            const f32x2 pp = pack2(pv[b][h * T + tt], pv[b][h * T + tt]);
#pragma unroll
            for (int j = 0; j < NP; ++j) o2[h][j] = ffma2(pp, v2[j], o2[h][j]);
          }
        }
      }
      con_slot = con_slot + 1 == NS ? 0 : con_slot + 1;
      con_phase ^= (con_slot == 0);
      --inflight;
      __syncwarp();
      top_up();
    }

    // ---- merge the 4 lane groups of the warp (shuffles) ----------------
    // l per head: the sum over the T lanes of the head within the group
    float lsum = l_own;
#pragma unroll
    for (int off = 1; off < T; off <<= 1) lsum += __shfl_xor_sync(FULL_MASK, lsum, off);
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      const float lh = __shfl_sync(FULL_MASK, lsum, gbase | (h * T));
      float M = m_all[h];
      M = fmaxf(M, __shfl_xor_sync(FULL_MASK, M, 8));
      M = fmaxf(M, __shfl_xor_sync(FULL_MASK, M, 16));
      const float w = fast_exp2(m_all[h] - M);
      float L = lh * w;
      L += __shfl_xor_sync(FULL_MASK, L, 8);
      L += __shfl_xor_sync(FULL_MASK, L, 16);
      const f32x2 w2 = pack2(w, w);
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        float2 v = unpack2(fmul2(o2[h][j], w2));
        v.x += __shfl_xor_sync(FULL_MASK, v.x, 8);
        v.y += __shfl_xor_sync(FULL_MASK, v.y, 8);
        v.x += __shfl_xor_sync(FULL_MASK, v.x, 16);
        v.y += __shfl_xor_sync(FULL_MASK, v.y, 16);
        o2[h][j] = pack2(v.x, v.y);
      }
      if (grp == 0 && li == 0) red_ml[warp * GP + h] = make_float2(M, L);
    }
    if (grp == 0) {
#pragma unroll
      for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          float4 *dst = reinterpret_cast<float4 *>(red_o + (warp * GP + h) * D + (li + 8 * c) * 8);
          const float2 a0 = unpack2(o2[h][4 * c + 0]), a1 = unpack2(o2[h][4 * c + 1]);
          const float2 a2 = unpack2(o2[h][4 * c + 2]), a3 = unpack2(o2[h][4 * c + 3]);
          dst[0] = make_float4(a0.x, a0.y, a1.x, a1.y);
          dst[1] = make_float4(a2.x, a2.y, a3.x, a3.y);
        }
    }
    if (tid == 0) s_unit[(ordinal + 2) & 3] = next_id;
    named_barrier_sync();

    // ---- merge the 4 warps into the split's partial (m, l, o) ----------
    const int64_t bh0 = (int64_t)cur.b * Hq + cur.h0;
    for (int idx = tid; idx < (cur.bad ? 0 : cur.nh * D); idx += ATTN_THREADS) {
      const int h = idx / D, d = idx % D;
      float M = ATTN_NEG;
#pragma unroll
      for (int w = 0; w < ATTN_WARPS; ++w) M = fmaxf(M, red_ml[w * GP + h].x);
      float L = 0.0f, O = 0.0f;
#pragma unroll
      for (int w = 0; w < ATTN_WARPS; ++w) {
        const float2 ml = red_ml[w * GP + h];
        const float wt = fast_exp2(ml.x - M);
        L = fmaf(ml.y, wt, L);
        O = fmaf(red_o[(w * GP + h) * D + d], wt, O);
      }
      const int64_t ps = (bh0 + h) * a.nsplit_max + cur.split;
      a.ws_o[ps * D + d] = O;
      if (d == 0) a.ws_ml[ps] = make_float2(M, L);
    }
    // rotate units; the barrier also protects red_o / red_ml
    named_barrier_sync();
    ++ordinal;
    cur = nxt;
    cur_cnt = nxt_cnt;
    pid_cur = pid_nxt;
    nxt = decode_unit(a, s_unit[(ordinal + 1) & 3], GP, total_units, s_full, rs, seq);
    nxt_cnt = warp_pages(nxt, warp);
    pid_nxt = load_pids(nxt, nxt_cnt);
    stage_q(nxt, (ordinal + 1) & 1);
    if (iss_u == 1) {
      iss_u = 0;  // pages already issued of the old "next" unit belong to "cur" now
    } else {
      iss_i = 0;  // the warp had issued nothing of the old "next" unit
    }
  }
  if (dead) {
    // let the copies still in flight land before the CTA's shared memory goes
    for (int k = 0; k < inflight; ++k) {
      (void)mbar_wait(&wbars[con_slot], con_phase, 100000000ull);
      con_slot = con_slot + 1 == NS ? 0 : con_slot + 1;
      con_phase ^= (con_slot == 0);
    }
  }
}

// Fold each active row's split partials: out = sum_s w_s o_s / sum_s w_s l_s
// with w_s = 2^(m_s - max m).  One CTA per (row, q head); its 4 warps take
// every 4th split (a fixed assignment, so the result is deterministic), each
// lane a float vector of dims.  A warp issues the loads of up to 16 of its
// splits at once and folds them with one rescale; the 4 warps then combine
// through shared memory.  Padding and rejected rows get zeros and
// lse = -inf.
template <int D>
__global__ void __launch_bounds__(ATTN_THREADS) attn_merge_kernel(const AttnArgs a) {
  constexpr int VEC = D / 32;  // dims per lane
  constexpr int BLK = 16;      // splits in flight per warp
  __shared__ float s_m[ATTN_WARPS], s_l[ATTN_WARPS];
  __shared__ __align__(16) float s_o[ATTN_WARPS][D];
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The lengths and flags were final before the persistent grid started
  // (its CTAs let this grid start only after their own wait), so they are
  // read before this grid's wait; the partials only after it.
  const int64_t bh = (int64_t)b * a.num_qo_heads + h;
  const int n = a.seq_lens[b];
  const int act = a.active[b];
  pdl_wait();  // the partials of the persistent kernel
  pdl_trigger();
  // the persistent grid has completed: its unit counter starts again at zero
  // for the next call that runs on the same plan
  if (h == 0 && b == 0 && threadIdx.x == 0) a.plan->counter = 0;
  if (!act || n < 1 || (int64_t)n > a.max_tokens) {
    for (int d = threadIdx.x; d < D; d += ATTN_THREADS) store_out(a, bh * D + d, 0.0f);
    if (threadIdx.x == 0 && a.lse != nullptr) a.lse[bh] = -INFINITY;
    return;
  }
  const int npages = (n + ATTN_PAGE - 1) / ATTN_PAGE;
  const int nsplit = (npages + ATTN_PAGES_PER_SPLIT - 1) / ATTN_PAGES_PER_SPLIT;
  const float2 *ml = a.ws_ml + bh * a.nsplit_max;
  const float *po = a.ws_o + bh * a.nsplit_max * D + lane * VEC;
  float M = ATTN_NEG, L = 0.0f, O[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) O[e] = 0.0f;
  for (int s0 = w; s0 < nsplit; s0 += ATTN_WARPS * BLK) {
    float2 v[BLK];
    float o[BLK][VEC];
#pragma unroll
    for (int k = 0; k < BLK; ++k) {
      const int s = s0 + k * ATTN_WARPS;
      v[k] = make_float2(ATTN_NEG, 0.0f);
#pragma unroll
      for (int e = 0; e < VEC; ++e) o[k][e] = 0.0f;
      if (s < nsplit) {
        v[k] = ml[s];
        if constexpr (VEC == 4) {
          const float4 t = *reinterpret_cast<const float4 *>(po + (int64_t)s * D);
          o[k][0] = t.x, o[k][1] = t.y, o[k][2] = t.z, o[k][3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2 *>(po + (int64_t)s * D);
          o[k][0] = t.x, o[k][1] = t.y;
        }
      }
    }
    float mb = M;
#pragma unroll
    for (int k = 0; k < BLK; ++k) mb = fmaxf(mb, v[k].x);
    const float sc = fast_exp2(M - mb);
    L *= sc;
#pragma unroll
    for (int e = 0; e < VEC; ++e) O[e] *= sc;
#pragma unroll
    for (int k = 0; k < BLK; ++k) {
      const float wt = fast_exp2(v[k].x - mb);
      L = fmaf(v[k].y, wt, L);
#pragma unroll
      for (int e = 0; e < VEC; ++e) O[e] = fmaf(o[k][e], wt, O[e]);
    }
    M = mb;
  }
  if (lane == 0) {
    s_m[w] = M;
    s_l[w] = L;
  }
#pragma unroll
  for (int e = 0; e < VEC; ++e) s_o[w][lane * VEC + e] = O[e];
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += ATTN_THREADS) {
    float Mx = ATTN_NEG;
#pragma unroll
    for (int k = 0; k < ATTN_WARPS; ++k) Mx = fmaxf(Mx, s_m[k]);
    float Lt = 0.0f, Ot = 0.0f;
#pragma unroll
    for (int k = 0; k < ATTN_WARPS; ++k) {
      const float wt = fast_exp2(s_m[k] - Mx);
      Lt = fmaf(s_l[k], wt, Lt);
      Ot = fmaf(s_o[k][d], wt, Ot);
    }
    store_out(a, bh * D + d, Ot / Lt);
    if (d == 0 && a.lse != nullptr) a.lse[bh] = (Mx + log2f(Lt)) * LN2;
  }
}

// q heads per CTA: the group rounded up to 2 / 4 / 8, at most 4 for
// head_dim 128 (8 would not fit the registers); larger groups use several
// q-head blocks per kv head.
static int heads_per_cta(int D, int group) {
  const int cap = D == 128 ? 4 : 8;
  const int gp = group <= 2 ? 2 : (group <= 4 ? 4 : 8);
  return gp < cap ? gp : cap;
}

// what a call launches: the planner, the attention kernels, or both
enum AttnMode { ATTN_PLAN_AND_RUN = 0, ATTN_PLAN_ONLY = 1, ATTN_RUN_ONLY = 2 };

template <int D, int GP, int NS>
static int launch_attn(const AttnArgs &a, const CUtensorMap &tmap, cudaStream_t st,
                       AttnMode mode) {
  using S = AttnShape<D, GP, NS>;
  auto kern = attn_persistent_kernel<D, GP, NS>;
  // persistent grid per device (0: not known yet); host threads may race to
  // fill a slot, and all write the same value
  static std::atomic<int> grid_for_device[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  int grid = grid_for_device[dev & 63].load(std::memory_order_acquire);
  if (grid == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, ATTN_THREADS,
                                                      S::SMEM_BYTES) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (per_sm < 1) return PKV_ERR_UNSUPPORTED;
    grid = sms * per_sm;
    grid_for_device[dev & 63].store(grid, std::memory_order_release);
  }
  if (mode != ATTN_RUN_ONLY &&
      launch_pdl(attn_plan_kernel, dim3(1), dim3(PLAN_THREADS), 0, st, a) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (mode == ATTN_PLAN_ONLY) return launch_status();
  if (launch_pdl(kern, dim3(grid), dim3(ATTN_THREADS), S::SMEM_BYTES, st, a, tmap) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (launch_pdl(attn_merge_kernel<D>, dim3((unsigned)a.num_qo_heads, (unsigned)a.batch),
                 dim3(ATTN_THREADS), 0, st, a) != cudaSuccess)
    return PKV_ERR_CUDA;
  return launch_status();
}

template <int D>
static int dispatch_gp(const AttnArgs &a, const CUtensorMap &tmap, cudaStream_t st,
                       AttnMode mode) {
  constexpr int NS = D == 128 ? 3 : 6;
  switch (a.gp) {
    case 2: return launch_attn<D, 2, NS>(a, tmap, st, mode);
    case 4: return launch_attn<D, 4, NS>(a, tmap, st, mode);
    default:
      if constexpr (D == 64) return launch_attn<D, 8, NS>(a, tmap, st, mode);
      return PKV_ERR_UNSUPPORTED;
  }
}

// The driver's tensor-map encoder, fetched once through the runtime (no
// link-time dependency on libcuda).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// 5-D view of the whole cache for the TMA engine, innermost first:
// (head_dim, kv head, slot, K/V, layer * num_pages + page).  One box is one
// 16-token block of one page and kv head: head_dim x 1 x 16 x 2 x 1.
static int encode_cache_map(CUtensorMap *map, const void *cache, const pkv_cache_t *g) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return PKV_ERR_CUDA;
  const cuuint64_t D = (cuuint64_t)g->head_dim, H = (cuuint64_t)g->num_kv_heads;
  const cuuint64_t PS = (cuuint64_t)g->page_size;
  const cuuint64_t dims[5] = {D, H, PS, 2, (cuuint64_t)g->num_layers * (cuuint64_t)g->num_pages};
  const cuuint64_t strides[4] = {D * 2, H * D * 2, PS * H * D * 2, 2 * PS * H * D * 2};
  const cuuint32_t box[5] = {(cuuint32_t)D, 1, (cuuint32_t)ATTN_PAGE, 2, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(cache), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_UNSUPPORTED;
}

// splits of the longest possible row (max_tokens = max_pages * page_size)
static size_t nsplit_for(int64_t max_tokens) {
  const int64_t blocks = (max_tokens + ATTN_PAGE - 1) / ATTN_PAGE;
  return (size_t)((blocks + ATTN_PAGES_PER_SPLIT - 1) / ATTN_PAGES_PER_SPLIT);
}

struct WsLayout {
  size_t o, ml, row_start, plan, total;
};

static WsLayout ws_layout(int batch, int num_qo_heads, int head_dim, int64_t max_tokens) {
  WsLayout w;
  const size_t units = (size_t)batch * num_qo_heads * nsplit_for(max_tokens);
  w.o = 0;
  w.ml = align_up(units * head_dim * sizeof(float), 256);
  w.row_start = w.ml + align_up(units * sizeof(float2), 256);
  w.plan = w.row_start + align_up((size_t)(2 * batch + 1) * sizeof(int32_t), 256);
  w.total = w.plan + 256;
  return w;
}

}  // namespace pkv

extern "C" size_t pkv_decode_workspace_bytes(int batch, int num_qo_heads, int head_dim,
                                             int max_pages, int page_size) {
  using namespace pkv;
  if (batch <= 0 || num_qo_heads <= 0 || head_dim <= 0 || max_pages <= 0 || page_size <= 0)
    return 0;
  return ws_layout(batch, num_qo_heads, head_dim, (int64_t)max_pages * page_size).total;
}

namespace pkv {

// Checks a call's arguments other than the workspace; *ws_need gets the
// workspace bytes the call needs.  With plan_only the call has no cache, q
// or output (the planner reads none).
static int attn_check(const pkv_cache_t *geom, const void *cache, int layer, const void *q,
                      int num_qo_heads, float sm_scale, const int32_t *page_table, int max_pages,
                      const int32_t *seq_lens, const int32_t *active, int batch, const void *out,
                      bool plan_only, size_t *ws_need) {
  const int st = check_geometry(geom);
  if (st != PKV_OK) return st;
  if (!seq_lens || !active) return PKV_ERR_INVALID_ARG;
  if (!plan_only && (!cache || !q || !page_table || !out)) return PKV_ERR_INVALID_ARG;
  if (batch <= 0 || max_pages <= 0 || layer < 0 || layer >= geom->num_layers ||
      num_qo_heads <= 0 || num_qo_heads % geom->num_kv_heads != 0)
    return PKV_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return PKV_ERR_INVALID_ARG;  // NaN
  const int D = geom->head_dim;
  const int group = num_qo_heads / geom->num_kv_heads;
  if ((D != 64 && D != 128) || geom->page_size % ATTN_PAGE != 0 ||
      geom->page_size > ATTN_MAX_PAGE_SIZE || group > 64)
    return PKV_ERR_UNSUPPORTED;
  const int64_t max_tokens = (int64_t)max_pages * geom->page_size;
  if (max_tokens > INT32_MAX ||
      (int64_t)batch * num_qo_heads * (int64_t)nsplit_for(max_tokens) > (1ll << 30) ||
      (int64_t)geom->num_pages * (geom->page_size / ATTN_PAGE) > INT32_MAX)
    return PKV_ERR_UNSUPPORTED;
  if (!plan_only && (!aligned16(cache) || !aligned16(q))) return PKV_ERR_INVALID_ARG;
  if ((int64_t)geom->num_layers * geom->num_pages > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  *ws_need = ws_layout(batch, num_qo_heads, D, max_tokens).total;
  return PKV_OK;
}

// Checks a call's arguments and fills the kernels' arguments.
static int attn_setup(const pkv_cache_t *geom, const void *cache, int layer, const void *q,
                      int num_qo_heads, float sm_scale, const int32_t *page_table, int max_pages,
                      const int32_t *seq_lens, const int32_t *active, int batch, void *out,
                      int out_fp32, float *lse, void *workspace, size_t workspace_bytes,
                      int32_t *err_word, bool plan_only, AttnArgs *pa, CUtensorMap *tmap) {
  size_t need = 0;
  int st = attn_check(geom, cache, layer, q, num_qo_heads, sm_scale, page_table, max_pages,
                      seq_lens, active, batch, out, plan_only, &need);
  if (st != PKV_OK) return st;
  if (workspace == nullptr || workspace_bytes < need) return PKV_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return PKV_ERR_INVALID_ARG;
  const int D = geom->head_dim;
  const int group = num_qo_heads / geom->num_kv_heads;
  const int64_t max_tokens = (int64_t)max_pages * geom->page_size;
  const WsLayout wl = ws_layout(batch, num_qo_heads, D, max_tokens);

  AttnArgs &a = *pa;
  const int64_t row_bytes = (int64_t)D * 2;
  a.cache = static_cast<const unsigned char *>(cache);
  a.tok_stride = row_bytes * geom->num_kv_heads;
  a.kv_stride = a.tok_stride * geom->page_size;
  a.page_stride = a.kv_stride * 2;
  a.layer_off = a.page_stride * (int64_t)geom->num_pages * layer;
  a.num_pages = geom->num_pages;
  a.num_kv_heads = geom->num_kv_heads;
  a.head_dim = D;
  a.q = static_cast<const uint16_t *>(q);
  a.num_qo_heads = num_qo_heads;
  a.group = group;
  a.gp = heads_per_cta(D, group);
  a.qblocks = (group + a.gp - 1) / a.gp;
  a.qscale = sm_scale * LOG2E;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.bpp = geom->page_size / ATTN_PAGE;
  a.max_tokens = max_tokens;
  a.seq_lens = seq_lens;
  a.active = active;
  a.batch = batch;
  a.out = out;
  a.out_fp32 = out_fp32 != 0;
  a.lse = lse;
  a.nsplit_max = (int)nsplit_for(max_tokens);
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  a.ws_o = reinterpret_cast<float *>(ws + wl.o);
  a.ws_ml = reinterpret_cast<float2 *>(ws + wl.ml);
  a.row_start = reinterpret_cast<int32_t *>(ws + wl.row_start);
  a.part_rows = a.row_start + batch + 1;
  a.plan = reinterpret_cast<PlanHeader *>(ws + wl.plan);
  a.err = err_word;
  a.layer = layer;
  if (!plan_only) {
    st = encode_cache_map(tmap, cache, geom);
    if (st != PKV_OK) return st;
  }
  return PKV_OK;
}

static int attn_call(const pkv_cache_t *geom, const void *cache, int layer, const void *q,
                     int num_qo_heads, float sm_scale, const int32_t *page_table, int max_pages,
                     const int32_t *seq_lens, const int32_t *active, int batch, void *out,
                     int out_fp32, float *lse, void *workspace, size_t workspace_bytes,
                     int32_t *err_word, void *stream, AttnMode mode) {
  AttnArgs a;
  alignas(64) CUtensorMap tmap;
  memset(&tmap, 0, sizeof(tmap));
  const int st = attn_setup(geom, cache, layer, q, num_qo_heads, sm_scale, page_table, max_pages,
                            seq_lens, active, batch, out, out_fp32, lse, workspace,
                            workspace_bytes, err_word, mode == ATTN_PLAN_ONLY, &a, &tmap);
  if (st != PKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return a.head_dim == 128 ? dispatch_gp<128>(a, tmap, s, mode) : dispatch_gp<64>(a, tmap, s, mode);
}

}  // namespace pkv

extern "C" int pkv_paged_decode_attn(const pkv_cache_t *geom, const void *cache, int layer,
                                     const void *q, int num_qo_heads, float sm_scale,
                                     const int32_t *page_table, int max_pages,
                                     const int32_t *seq_lens, const int32_t *active, int batch,
                                     void *out, int out_fp32, float *lse, void *workspace,
                                     size_t workspace_bytes, int32_t *err_word, void *stream) {
  return pkv::attn_call(geom, cache, layer, q, num_qo_heads, sm_scale, page_table, max_pages,
                        seq_lens, active, batch, out, out_fp32, lse, workspace, workspace_bytes,
                        err_word, stream, pkv::ATTN_PLAN_AND_RUN);
}

extern "C" int pkv_decode_plan(const pkv_cache_t *geom, int num_qo_heads, int max_pages,
                               const int32_t *seq_lens, const int32_t *active, int batch,
                               void *workspace, size_t workspace_bytes, int32_t *err_word,
                               void *stream) {
  return pkv::attn_call(geom, nullptr, 0, nullptr, num_qo_heads, 1.0f, nullptr, max_pages,
                        seq_lens, active, batch, nullptr, 0, nullptr, workspace, workspace_bytes,
                        err_word, stream, pkv::ATTN_PLAN_ONLY);
}

extern "C" int pkv_paged_decode_attn_planned(const pkv_cache_t *geom, const void *cache, int layer,
                                             const void *q, int num_qo_heads, float sm_scale,
                                             const int32_t *page_table, int max_pages,
                                             const int32_t *seq_lens, const int32_t *active,
                                             int batch, void *out, int out_fp32, float *lse,
                                             void *workspace, size_t workspace_bytes,
                                             int32_t *err_word, void *stream) {
  return pkv::attn_call(geom, cache, layer, q, num_qo_heads, sm_scale, page_table, max_pages,
                        seq_lens, active, batch, out, out_fp32, lse, workspace, workspace_bytes,
                        err_word, stream, pkv::ATTN_RUN_ONLY);
}

// ---------------------------------------------------------------------------
// Static-scratch variant: the same kernels, with their scratch in a
// file-scope device array instead of a caller-provided workspace.
// ---------------------------------------------------------------------------
namespace pkv {

// Every device that loads the library holds this array until the process
// exits.  The kernels need nothing in it to start at zero: the planner
// rewrites the split table and the unit counter on every call and each
// partial is written before it is read.
static __device__ __align__(256) unsigned char g_attn_scratch[PKV_ATTN_STATIC_SCRATCH_BYTES];

// Device address of the array in each CUDA context that has used it.  The
// host-side name is only a stand-in for that address, and a context that is
// destroyed and made again (cudaDeviceReset) loads the module anew, possibly
// at another address: the cache is keyed by the driver's context id, which
// is never reused within a process.  Host threads share it under a mutex.
struct ScratchAddr {
  unsigned long long ctx_id;
  void *ptr;
};
constexpr int SCRATCH_CTX_SLOTS = 64;
static std::mutex g_scratch_mu;
static ScratchAddr g_scratch_addr[SCRATCH_CTX_SLOTS];
static int g_scratch_used = 0;

static int current_context_id(unsigned long long *id) {
  static const auto fns = []() {
    std::pair<PFN_cuCtxGetCurrent_v4000, PFN_cuCtxGetId_v12000> f{nullptr, nullptr};
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.first = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.second = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    return f;
  }();
  if (fns.first == nullptr || fns.second == nullptr) return PKV_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (fns.first(&ctx) != CUDA_SUCCESS || ctx == nullptr) return PKV_ERR_CUDA;
  return fns.second(ctx, id) == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

// Device address of the array in the current context (the current device's
// context), looked up with cudaGetSymbolAddress the first time a context
// uses it.
static int static_scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = 0;
  if (current_context_id(&id) == PKV_OK) {
    for (int i = 0; i < g_scratch_used; ++i)
      if (g_scratch_addr[i].ctx_id == id) {
        *out = g_scratch_addr[i].ptr;
        return PKV_OK;
      }
  }
  // first use in this context: the lookup also makes the runtime's context
  // of the device current if no call has done so yet
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_attn_scratch) != cudaSuccess || ptr == nullptr)
    return PKV_ERR_CUDA;
  if (current_context_id(&id) != PKV_OK) return PKV_ERR_CUDA;
  const int slot = g_scratch_used < SCRATCH_CTX_SLOTS ? g_scratch_used++
                                                      : (int)(id % SCRATCH_CTX_SLOTS);
  g_scratch_addr[slot] = ScratchAddr{id, ptr};
  *out = ptr;
  return PKV_OK;
}

}  // namespace pkv

extern "C" int pkv_paged_decode_attn_static(const pkv_cache_t *geom, const void *cache, int layer,
                                            const void *q, int num_qo_heads, float sm_scale,
                                            const int32_t *page_table, int max_pages,
                                            const int32_t *seq_lens, const int32_t *active,
                                            int batch, void *out, int out_fp32, float *lse,
                                            int32_t *err_word, void *stream) {
  using namespace pkv;
  // every argument check first, so that the status names what is wrong with
  // the call whatever its size; then the size against the array
  size_t need = 0;
  int st = attn_check(geom, cache, layer, q, num_qo_heads, sm_scale, page_table, max_pages,
                      seq_lens, active, batch, out, false, &need);
  if (st != PKV_OK) return st;
  if (need > (size_t)PKV_ATTN_STATIC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  void *scratch = nullptr;
  st = static_scratch_address(&scratch);
  if (st != PKV_OK) return st;
  return pkv_paged_decode_attn(geom, cache, layer, q, num_qo_heads, sm_scale, page_table,
                               max_pages, seq_lens, active, batch, out, out_fp32, lse, scratch,
                               (size_t)PKV_ATTN_STATIC_SCRATCH_BYTES, err_word, stream);
}
