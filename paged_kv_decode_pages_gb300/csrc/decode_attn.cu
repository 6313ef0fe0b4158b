// decode_attn.cu -- grouped-query decode attention over the paged cache:
// attn_wrapper.run(q, kv_cache) of "Adding a Model" (vox-serve docs),
// section "1. The model code", for the layout
// [num_layers, num_pages, 2, page_size, num_kv_heads, head_dim].
//
// Design (HBM-bound; CUDA cores, no tensor cores):
//  * split-KV: a row's pages are cut into fixed 32-page (512-token) splits;
//    one CTA per (kv head, q-head block, split, row).  The split size does
//    not depend on the batch, so a row's result depends on its inputs only.
//  * each of the CTA's 4 warps streams its own pages (round-robin) through
//    its own ring of NS shared-memory stages; a stage is one page of one kv
//    head: 16 K rows + 16 V rows, each row head_dim bf16 contiguous in HBM,
//    brought in by 32 bulk async copies (cp.async.bulk, the TMA engine) that
//    complete on the stage's mbarrier.  Waits are bounded.
//  * GQA sharing: the warp holds the q of all the group's heads in
//    registers, so every K / V element is read from shared memory and
//    converted once and used for every head of the group.
//  * lanes: 8 lanes share one token, each lane owns head_dim/8 dims, read as
//    16-byte vectors (conflict-free); q.k partial sums are summed over the
//    8 lanes with 3 xor-shuffles; the online softmax runs in the log2
//    domain with a lazy maximum (rescale only when a score exceeds the
//    running maximum by more than 8).
//  * the 4 groups x 4 warps of a CTA merge through shared memory; a row with
//    one split writes its output directly, longer rows write (m, l, o)
//    partials that a merge kernel folds in split order.
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int ATTN_WARPS = 4;
constexpr int ATTN_PAGES_PER_SPLIT = 32;
constexpr int ATTN_PAGE = 16;
constexpr float ATTN_TAU = 8.0f;       // lazy-rescale threshold (log2 units)
constexpr float ATTN_NEG = -1.0e30f;   // "no score yet" (finite: keeps 2^(s-m) at 0)
constexpr float LN2 = 0.69314718055994530942f;
constexpr float LOG2E = 1.44269504088896340736f;

struct AttnArgs {
  const unsigned char *cache;  // byte address of the cache
  int64_t layer_off;           // bytes
  int64_t page_stride;         // bytes
  int64_t kv_stride;           // bytes
  int64_t tok_stride;          // bytes
  int num_pages;
  int num_kv_heads;
  const uint16_t *q;           // [B][Hq][D] bf16 bits
  int num_qo_heads;
  int group;                   // Hq / Hkv
  int qblocks;                 // q-head blocks per kv head
  float qscale;                // sm_scale * log2(e)
  const int32_t *page_table;
  int max_pages;
  const int32_t *seq_lens;
  const int32_t *active;
  int batch;
  void *out;
  int out_fp32;
  float *lse;
  float *ws_o;                 // [B][Hq][nsplit_max][D]
  float2 *ws_ml;               // [B][Hq][nsplit_max]
  int nsplit_max;
  int32_t *err;
};

template <int D>
__device__ __forceinline__ void store_out(const AttnArgs &a, int64_t idx, float v) {
  if (a.out_fp32)
    static_cast<float *>(a.out)[idx] = v;
  else
    static_cast<uint16_t *>(a.out)[idx] = (uint16_t)f32_to_bf16_bits(v);
}

template <int D, int GP, int NS>
struct AttnShape {
  static constexpr int T = 8 / GP;              // tokens per lane group per batch
  static constexpr int TOK_PER_BATCH = 4 * T;   // tokens per warp per batch
  static constexpr int BATCHES = ATTN_PAGE / TOK_PER_BATCH;
  static constexpr int DPL = D / 8;             // dims per lane
  static constexpr int NCH = DPL / 8;           // 16-byte chunks per lane per row
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int STAGE_BYTES = 2 * ATTN_PAGE * ROW_BYTES;
  static constexpr int RING_BYTES = ATTN_WARPS * NS * STAGE_BYTES;
  static constexpr int RED_BYTES = ATTN_WARPS * 4 * GP * (D * 4 + 8);
  static constexpr int DATA_BYTES = RING_BYTES > RED_BYTES ? RING_BYTES : RED_BYTES;
  static constexpr int SMEM_BYTES = DATA_BYTES + ATTN_WARPS * NS * 8;
  static_assert(GP == 2 || GP == 4 || GP == 8, "GP");
  static_assert(D == 64 || D == 128, "D");
};

template <int D, int GP, int NS>
__global__ void __launch_bounds__(ATTN_WARPS * 32, 2) attn_split_kernel(const AttnArgs a) {
  using S = AttnShape<D, GP, NS>;
  constexpr int T = S::T, DPL = S::DPL, NCH = S::NCH;

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::DATA_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = lane >> 3;
  const int li = lane & 7;

  const int b = blockIdx.z;
  const int split = blockIdx.y;
  const int g = blockIdx.x / a.qblocks;
  const int qb = blockIdx.x % a.qblocks;
  const int h0 = g * a.group + qb * GP;
  const int nh = min(GP, a.group - qb * GP);
  const int Hq = a.num_qo_heads;

  const bool act = a.active[b] != 0;
  const int n = act ? a.seq_lens[b] : 0;
  const bool bad_len = act && (n < 1 || (int64_t)n > (int64_t)a.max_pages * ATTN_PAGE);
  if (!act || bad_len) {
    // padding (or rejected) row: zeros, lse = -inf, written once by split 0
    if (split == 0) {
      for (int i = threadIdx.x; i < nh * D; i += blockDim.x)
        store_out<D>(a, ((int64_t)b * Hq + h0 + i / D) * D + i % D, 0.0f);
      if (a.lse != nullptr && threadIdx.x < nh) a.lse[(int64_t)b * Hq + h0 + threadIdx.x] = -INFINITY;
      if (bad_len && threadIdx.x == 0 && blockIdx.x == 0) report(a.err, PKV_DEV_ERR_SEQ_LEN);
    }
    return;
  }
  const int npages = (n + ATTN_PAGE - 1) / ATTN_PAGE;
  const int nsplit = (npages + ATTN_PAGES_PER_SPLIT - 1) / ATTN_PAGES_PER_SPLIT;
  if (split >= nsplit) return;
  const int p_begin = split * ATTN_PAGES_PER_SPLIT;
  const int p_count = min(npages - p_begin, ATTN_PAGES_PER_SPLIT);
  const int my_count = p_count > warp ? (p_count - warp + ATTN_WARPS - 1) / ATTN_WARPS : 0;

  unsigned char *ring = smem + warp * NS * S::STAGE_BYTES;
  uint64_t *wbars = bars + warp * NS;
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&wbars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // q of the lane's dims for every head of the block, pre-scaled to log2 units
  float qf[GP][DPL];
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    if (h < nh) {
      const uint4 *qr = reinterpret_cast<const uint4 *>(a.q + ((int64_t)b * Hq + h0 + h) * D);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        float f[8];
        unpack8(__ldg(qr + li + 8 * c), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[h][8 * c + e] = f[e] * a.qscale;
      }
    } else {
#pragma unroll
      for (int d = 0; d < DPL; ++d) qf[h][d] = 0.0f;
    }
  }

  const unsigned char *head_base =
      a.cache + a.layer_off + (int64_t)g * S::ROW_BYTES;
  const int32_t *pt_row = a.page_table + (int64_t)b * a.max_pages;

  // issue the 32 row copies of the warp's i-th page into ring slot `slot`
  auto issue = [&](int i, int slot) {
    const int pi = p_begin + warp + i * ATTN_WARPS;
    int pid = __ldg(pt_row + pi);
    if (pid < 0 || pid >= a.num_pages) {
      if (lane == 0) report(a.err, PKV_DEV_ERR_PAGE);
      pid = 0;
    }
    uint64_t *bar = &wbars[slot];
    if (lane == 0) mbar_arrive_expect_tx(bar, S::STAGE_BYTES);
    __syncwarp();
    const int kv = lane >> 4;      // lanes 0-15: K rows, 16-31: V rows
    const int t = lane & 15;
    const unsigned char *src = head_base + (int64_t)pid * a.page_stride + kv * a.kv_stride +
                               (int64_t)t * a.tok_stride;
    unsigned char *dst = ring + slot * S::STAGE_BYTES + (kv * ATTN_PAGE + t) * S::ROW_BYTES;
    bulk_copy_g2s(dst, src, S::ROW_BYTES, bar);
  };

  float o[GP][DPL];
  float m[GP], l[GP];
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    m[h] = ATTN_NEG;
    l[h] = 0.0f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[h][d] = 0.0f;
  }

  const int prologue = my_count < NS ? my_count : NS;
  for (int i = 0; i < prologue; ++i) issue(i, i);

  bool timed_out = false;
  int consumed = 0;
  for (int i = 0; i < my_count; ++i) {
    const int slot = i % NS;
    // the give-up decision must be warp-uniform: the shuffles below need all lanes
    const bool landed = mbar_wait(&wbars[slot], (uint32_t)((i / NS) & 1));
    if (!__all_sync(FULL_MASK, landed)) {
      timed_out = true;
      break;
    }
    consumed = i + 1;
    const unsigned char *kst = ring + slot * S::STAGE_BYTES;
    const unsigned char *vst = kst + ATTN_PAGE * S::ROW_BYTES;
    const int tok0 = (p_begin + warp + i * ATTN_WARPS) * ATTN_PAGE;
    const bool ragged = tok0 + ATTN_PAGE > n;

#pragma unroll
    for (int bt = 0; bt < S::BATCHES; ++bt) {
      const int tb = bt * S::TOK_PER_BATCH + grp * T;  // first token of this lane group
      float s[GP][T];
#pragma unroll
      for (int tt = 0; tt < T; ++tt) {
        const uint4 *kr = reinterpret_cast<const uint4 *>(kst + (tb + tt) * S::ROW_BYTES);
        float kf[DPL];
#pragma unroll
        for (int c = 0; c < NCH; ++c) unpack8(kr[li + 8 * c], kf + 8 * c);
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          float acc = 0.0f;
#pragma unroll
          for (int d = 0; d < DPL; ++d) acc = fmaf(qf[h][d], kf[d], acc);
          s[h][tt] = acc;
        }
      }
      // sum the partial dot products over the 8 lanes of the group
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) {
#pragma unroll
        for (int h = 0; h < GP; ++h)
#pragma unroll
          for (int tt = 0; tt < T; ++tt) s[h][tt] += __shfl_xor_sync(FULL_MASK, s[h][tt], off);
      }
      if (ragged) {
#pragma unroll
        for (int tt = 0; tt < T; ++tt)
          if (tok0 + tb + tt >= n) {
#pragma unroll
            for (int h = 0; h < GP; ++h) s[h][tt] = -INFINITY;
          }
      }
      // online softmax with a lazy maximum
      bool need = false;
#pragma unroll
      for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int tt = 0; tt < T; ++tt) need |= s[h][tt] > m[h] + ATTN_TAU;
      if (__any_sync(FULL_MASK, need)) {
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          float mx = s[h][0];
#pragma unroll
          for (int tt = 1; tt < T; ++tt) mx = fmaxf(mx, s[h][tt]);
          const float mn = fmaxf(m[h], mx);
          const float sc = fast_exp2(m[h] - mn);
          l[h] *= sc;
#pragma unroll
          for (int d = 0; d < DPL; ++d) o[h][d] *= sc;
          m[h] = mn;
        }
      }
      float p[GP][T];
#pragma unroll
      for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int tt = 0; tt < T; ++tt) {
          p[h][tt] = fast_exp2(s[h][tt] - m[h]);
          l[h] += p[h][tt];
        }
#pragma unroll
      for (int tt = 0; tt < T; ++tt) {
        const uint4 *vr = reinterpret_cast<const uint4 *>(vst + (tb + tt) * S::ROW_BYTES);
        float vf[DPL];
#pragma unroll
        for (int c = 0; c < NCH; ++c) unpack8(vr[li + 8 * c], vf + 8 * c);
        if (ragged && tok0 + tb + tt >= n) {
          // rows past the end of the sequence may hold any bits
#pragma unroll
          for (int d = 0; d < DPL; ++d) vf[d] = 0.0f;
        }
#pragma unroll
        for (int h = 0; h < GP; ++h)
#pragma unroll
          for (int d = 0; d < DPL; ++d) o[h][d] = fmaf(p[h][tt], vf[d], o[h][d]);
      }
    }
    __syncwarp();
    if (i + NS < my_count) {
      fence_proxy_async_smem();
      issue(i + NS, slot);
    }
  }
  if (timed_out) {
    if (lane == 0) report(a.err, PKV_DEV_ERR_TIMEOUT);
    // let the copies still in flight land before the shared memory is reused
    const int issued = my_count < consumed + NS ? my_count : consumed + NS;
    for (int i = consumed; i < issued; ++i)
      (void)mbar_wait(&wbars[i % NS], (uint32_t)((i / NS) & 1), 100000000ull);
  }

  // ---- merge the 16 lane groups of the CTA through shared memory --------
  __syncthreads();
  float *red_o = reinterpret_cast<float *>(smem);                              // [16][GP][D]
  float2 *red_ml = reinterpret_cast<float2 *>(smem + ATTN_WARPS * 4 * GP * D * 4);  // [16][GP]
  const int gi = warp * 4 + grp;
  if (li == 0) {
#pragma unroll
    for (int h = 0; h < GP; ++h) red_ml[gi * GP + h] = make_float2(m[h], l[h]);
  }
#pragma unroll
  for (int h = 0; h < GP; ++h)
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      float4 *dst = reinterpret_cast<float4 *>(red_o + (gi * GP + h) * D + (li + 8 * c) * 8);
      dst[0] = make_float4(o[h][8 * c + 0], o[h][8 * c + 1], o[h][8 * c + 2], o[h][8 * c + 3]);
      dst[1] = make_float4(o[h][8 * c + 4], o[h][8 * c + 5], o[h][8 * c + 6], o[h][8 * c + 7]);
    }
  __syncthreads();

  for (int idx = threadIdx.x; idx < nh * D; idx += blockDim.x) {
    const int h = idx / D, d = idx % D;
    float M = ATTN_NEG;
#pragma unroll
    for (int q = 0; q < ATTN_WARPS * 4; ++q) M = fmaxf(M, red_ml[q * GP + h].x);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int q = 0; q < ATTN_WARPS * 4; ++q) {
      const float2 ml = red_ml[q * GP + h];
      const float w = fast_exp2(ml.x - M);
      L = fmaf(ml.y, w, L);
      O = fmaf(red_o[(q * GP + h) * D + d], w, O);
    }
    const int64_t bh = (int64_t)b * Hq + h0 + h;
    if (nsplit == 1) {
      store_out<D>(a, bh * D + d, O / L);
      if (d == 0 && a.lse != nullptr) a.lse[bh] = (M + log2f(L)) * LN2;
    } else {
      const int64_t ps = bh * a.nsplit_max + split;
      a.ws_o[ps * D + d] = O;
      if (d == 0) a.ws_ml[ps] = make_float2(M, L);
    }
  }
}

// Fold the split partials of rows with more than one split, in split order.
template <int D>
__global__ void __launch_bounds__(D) attn_merge_kernel(const AttnArgs a) {
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int d = threadIdx.x;
  if (!a.active[b]) return;
  const int n = a.seq_lens[b];
  if (n < 1 || (int64_t)n > (int64_t)a.max_pages * ATTN_PAGE) return;
  const int npages = (n + ATTN_PAGE - 1) / ATTN_PAGE;
  const int nsplit = (npages + ATTN_PAGES_PER_SPLIT - 1) / ATTN_PAGES_PER_SPLIT;
  if (nsplit <= 1) return;
  const int64_t bh = (int64_t)b * a.num_qo_heads + h;
  const float2 *ml = a.ws_ml + bh * a.nsplit_max;
  const float *po = a.ws_o + bh * a.nsplit_max * D + d;
  float M = ATTN_NEG;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ml[s].x);
  float L = 0.0f, O = 0.0f;
  for (int s = 0; s < nsplit; ++s) {
    const float2 v = ml[s];
    const float w = fast_exp2(v.x - M);
    L = fmaf(v.y, w, L);
    O = fmaf(po[(int64_t)s * D], w, O);
  }
  store_out<D>(a, bh * D + d, O / L);
  if (d == 0 && a.lse != nullptr) a.lse[bh] = (M + log2f(L)) * LN2;
}

template <int D, int GP, int NS>
static int launch_attn(const AttnArgs &a, int hkv, cudaStream_t st) {
  using S = AttnShape<D, GP, NS>;
  auto kern = attn_split_kernel<D, GP, NS>;
  static unsigned long long configured = 0;  // one bit per device; a race only repeats the call
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    configured |= bit;
  }
  dim3 grid((unsigned)(hkv * a.qblocks), (unsigned)a.nsplit_max, (unsigned)a.batch);
  kern<<<grid, ATTN_WARPS * 32, S::SMEM_BYTES, st>>>(a);
  int rc = launch_status();
  if (rc != PKV_OK) return rc;
  if (a.nsplit_max > 1) {
    attn_merge_kernel<D><<<dim3((unsigned)a.num_qo_heads, (unsigned)a.batch), D, 0, st>>>(a);
    rc = launch_status();
  }
  return rc;
}

// q heads per CTA: the group rounded up to 2 / 4 / 8, at most 4 for
// head_dim 128 (8 would not fit the registers); larger groups use several
// q-head blocks per kv head.
static int heads_per_cta(int D, int group) {
  const int cap = D == 128 ? 4 : 8;
  const int gp = group <= 2 ? 2 : (group <= 4 ? 4 : 8);
  return gp < cap ? gp : cap;
}

template <int D>
static int dispatch_gp(const AttnArgs &a, int hkv, int gp, cudaStream_t st) {
  constexpr int NS = D == 128 ? 3 : 6;
  switch (gp) {
    case 2: return launch_attn<D, 2, NS>(a, hkv, st);
    case 4: return launch_attn<D, 4, NS>(a, hkv, st);
    default:
      if constexpr (D == 64) return launch_attn<D, 8, NS>(a, hkv, st);
      return PKV_ERR_UNSUPPORTED;
  }
}

static size_t nsplit_for(int max_pages) {
  return (size_t)((max_pages + ATTN_PAGES_PER_SPLIT - 1) / ATTN_PAGES_PER_SPLIT);
}

}  // namespace pkv

extern "C" size_t pkv_decode_workspace_bytes(int batch, int num_qo_heads, int head_dim,
                                             int max_pages, int page_size) {
  using namespace pkv;
  if (batch <= 0 || num_qo_heads <= 0 || head_dim <= 0 || max_pages <= 0 || page_size <= 0)
    return 0;
  const size_t ns = nsplit_for(max_pages);
  const size_t units = (size_t)batch * num_qo_heads * ns;
  return align_up(units * head_dim * sizeof(float), 256) + align_up(units * sizeof(float2), 256);
}

extern "C" int pkv_paged_decode_attn(const pkv_cache_t *geom, const void *cache, int layer,
                                     const void *q, int num_qo_heads, float sm_scale,
                                     const int32_t *page_table, int max_pages,
                                     const int32_t *seq_lens, const int32_t *active, int batch,
                                     void *out, int out_fp32, float *lse, void *workspace,
                                     size_t workspace_bytes, int32_t *err_word, void *stream) {
  using namespace pkv;
  int st = check_geometry(geom);
  if (st != PKV_OK) return st;
  if (!cache || !q || !page_table || !seq_lens || !active || !out) return PKV_ERR_INVALID_ARG;
  if (batch <= 0 || max_pages <= 0 || layer < 0 || layer >= geom->num_layers ||
      num_qo_heads <= 0 || num_qo_heads % geom->num_kv_heads != 0)
    return PKV_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return PKV_ERR_INVALID_ARG;  // NaN
  const int D = geom->head_dim;
  const int group = num_qo_heads / geom->num_kv_heads;
  if ((D != 64 && D != 128) || geom->page_size != ATTN_PAGE || group > 64)
    return PKV_ERR_UNSUPPORTED;
  if (batch > 65535 || nsplit_for(max_pages) > 65535) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(cache) || !aligned16(q)) return PKV_ERR_INVALID_ARG;
  const size_t need = pkv_decode_workspace_bytes(batch, num_qo_heads, D, max_pages, ATTN_PAGE);
  const int nsplit_max = (int)nsplit_for(max_pages);
  if (nsplit_max > 1 && (workspace == nullptr || workspace_bytes < need)) return PKV_ERR_WORKSPACE;
  if (workspace != nullptr && ((uintptr_t)workspace & 255u) != 0) return PKV_ERR_INVALID_ARG;

  AttnArgs a;
  const int64_t row_bytes = (int64_t)D * 2;
  a.cache = static_cast<const unsigned char *>(cache);
  a.tok_stride = row_bytes * geom->num_kv_heads;
  a.kv_stride = a.tok_stride * geom->page_size;
  a.page_stride = a.kv_stride * 2;
  a.layer_off = a.page_stride * (int64_t)geom->num_pages * layer;
  a.num_pages = geom->num_pages;
  a.num_kv_heads = geom->num_kv_heads;
  a.q = static_cast<const uint16_t *>(q);
  a.num_qo_heads = num_qo_heads;
  a.group = group;
  const int gp = heads_per_cta(D, group);
  a.qblocks = (group + gp - 1) / gp;
  a.qscale = sm_scale * LOG2E;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.active = active;
  a.batch = batch;
  a.out = out;
  a.out_fp32 = out_fp32 != 0;
  a.lse = lse;
  a.nsplit_max = nsplit_max;
  const size_t units = (size_t)batch * num_qo_heads * nsplit_max;
  a.ws_o = static_cast<float *>(workspace);
  a.ws_ml = workspace ? reinterpret_cast<float2 *>(static_cast<unsigned char *>(workspace) +
                                                   align_up(units * D * sizeof(float), 256))
                      : nullptr;
  a.err = err_word;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return D == 128 ? dispatch_gp<128>(a, geom->num_kv_heads, gp, s)
                  : dispatch_gp<64>(a, geom->num_kv_heads, gp, s);
}
