// kv_append.cu -- set_kv_cache of "Adding a Model" (vox-serve docs), section
// "1. The model code": each row's new K and V go to the page slot of
// position seq_len - 1 of layer `layer`; padding entries ("How a program
// runs") write their ignored values to the dummy page 0, slot 0.  The
// multi-token variant appends a prefill / mixed step's packed new tokens
// at positions seq_len - q .. seq_len - 1 of their requests.
//
// Bytes moved: per row 2 * num_kv_heads * head_dim * 2 read + the same
// written.  The kernels are gather-free scatters of 16-byte chunks: one warp
// per (row, K or V) -- the row's destination (owner request, page, slot) is
// found once per warp, and each lane moves every 32nd chunk of the row, all
// of its loads in flight at once; every store a full 16-byte vector.
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

struct AppendArgs {
  uint4 *cache;           // base of the whole cache, as 16-byte chunks
  int64_t layer_off;      // chunks
  int64_t page_stride;    // chunks
  int64_t kv_stride;      // chunks
  int64_t slot_stride;    // chunks
  int num_pages;
  int page_size;
  const uint4 *k;         // [B][row_chunks]
  const uint4 *v;
  int row_chunks;         // num_kv_heads * head_dim / 8
  const int32_t *page_table;
  int max_pages;
  const int32_t *seq_lens;
  const int32_t *active;
  int batch;
  int32_t *err;
};

constexpr int APPEND_THREADS = 256;

// one warp copies a row of row_chunks 16-byte chunks from src to dst
__device__ __forceinline__ void copy_row(uint4 *dst, const uint4 *src, int row_chunks, int lane) {
  int c = lane;
  for (; c + 96 < row_chunks; c += 128) {  // four chunks per lane in flight
    const uint4 x0 = __ldg(src + c), x1 = __ldg(src + c + 32);
    const uint4 x2 = __ldg(src + c + 64), x3 = __ldg(src + c + 96);
    dst[c] = x0;
    dst[c + 32] = x1;
    dst[c + 64] = x2;
    dst[c + 96] = x3;
  }
  for (; c < row_chunks; c += 32) dst[c] = __ldg(src + c);
}

__global__ void __launch_bounds__(APPEND_THREADS) kv_append_kernel(const AppendArgs a) {
  pdl_wait();
  pdl_trigger();  // the next kernel waits for this grid before reading the cache
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)a.batch * 2;
  const int64_t wstep = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < rows; w += wstep) {
    const int kv = (int)(w & 1);
    const int b = (int)(w >> 1);
    int64_t page = 0, slot = 0;
    if (a.active[b]) {
      const int n = a.seq_lens[b];
      if (n < 1 || (int64_t)n > (int64_t)a.max_pages * a.page_size) {
        if (lane == 0 && kv == 0) report(a.err, PKV_DEV_ERR_SEQ_LEN);
        continue;
      }
      const int pos = n - 1;
      page = a.page_table[(int64_t)b * a.max_pages + pos / a.page_size];
      slot = pos % a.page_size;
      if (page < 0 || page >= a.num_pages) {
        if (lane == 0 && kv == 0) report(a.err, PKV_DEV_ERR_PAGE);
        continue;
      }
    }
    copy_row(a.cache + a.layer_off + page * a.page_stride + kv * a.kv_stride + slot * a.slot_stride,
             (kv == 0 ? a.k : a.v) + (int64_t)b * a.row_chunks, a.row_chunks, lane);
  }
}

// ---------------------------------------------------------------------------
// multi-token append (prefill / mixed steps): token t of the packed rows
// belongs to the request b with qo_indptr[b] <= t < qo_indptr[b+1] and goes
// to position seq_len[b] - q_b + (t - qo_indptr[b])
// ---------------------------------------------------------------------------
struct AppendTokArgs {
  AppendArgs base;  // base.batch = requests; base.k / base.v = packed rows
  const int32_t *qo_indptr;
  int total_tokens;
};

__global__ void __launch_bounds__(256) kv_append_tokens_kernel(const AppendTokArgs t) {
  const AppendArgs &a = t.base;
  constexpr int SMEM_REQS = 1024;  // request tables up to this size are searched in shared memory
  __shared__ int32_t s_ind[SMEM_REQS + 1];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const bool in_smem = a.batch <= SMEM_REQS;
  if (in_smem) {
    for (int i = threadIdx.x; i <= a.batch; i += blockDim.x) s_ind[i] = __ldg(t.qo_indptr + i);
    __syncthreads();
  }
  const int32_t *ind = in_smem ? s_ind : t.qo_indptr;
  const int64_t rows = (int64_t)t.total_tokens * 2;
  const int64_t wstep = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < rows; w += wstep) {
    const int kv = (int)(w & 1);
    const int tok = (int)(w >> 1);
    // owner request: the last b with qo_indptr[b] <= tok
    int lo = 0, hi = a.batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ind[mid] <= tok)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int b = lo;
    const int first = ind[b], end = ind[b + 1];
    if (tok < first || tok >= end) {
      if (lane == 0 && kv == 0) report(a.err, PKV_DEV_ERR_INDPTR);
      continue;
    }
    int64_t page = 0, slot = 0;
    if (a.active[b]) {
      const int q = end - first;
      const int n = a.seq_lens[b];
      if (n < q || n < 1 || (int64_t)n > (int64_t)a.max_pages * a.page_size) {
        if (lane == 0 && kv == 0 && tok == first) report(a.err, PKV_DEV_ERR_SEQ_LEN);
        continue;
      }
      const int pos = n - q + (tok - first);
      page = a.page_table[(int64_t)b * a.max_pages + pos / a.page_size];
      slot = pos % a.page_size;
      if (page < 0 || page >= a.num_pages) {
        if (lane == 0 && kv == 0) report(a.err, PKV_DEV_ERR_PAGE);
        continue;
      }
    }
    copy_row(a.cache + a.layer_off + page * a.page_stride + kv * a.kv_stride + slot * a.slot_stride,
             (kv == 0 ? a.k : a.v) + (int64_t)tok * a.row_chunks, a.row_chunks, lane);
  }
}

}  // namespace pkv

extern "C" int pkv_kv_append(const pkv_cache_t *geom, void *cache, int layer, const void *k,
                             const void *v, const int32_t *page_table, int max_pages,
                             const int32_t *seq_lens, const int32_t *active, int batch,
                             int32_t *err_word, void *stream) {
  using namespace pkv;
  int st = check_geometry(geom);
  if (st != PKV_OK) return st;
  if (!cache || !k || !v || !page_table || !seq_lens || !active) return PKV_ERR_INVALID_ARG;
  if (batch <= 0 || max_pages <= 0 || layer < 0 || layer >= geom->num_layers)
    return PKV_ERR_INVALID_ARG;
  const int64_t row = (int64_t)geom->num_kv_heads * geom->head_dim;
  if (row % 8 != 0) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(cache) || !aligned16(k) || !aligned16(v)) return PKV_ERR_INVALID_ARG;

  AppendArgs a;
  a.cache = static_cast<uint4 *>(cache);
  a.slot_stride = row / 8;
  a.kv_stride = a.slot_stride * geom->page_size;
  a.page_stride = a.kv_stride * 2;
  a.layer_off = a.page_stride * (int64_t)geom->num_pages * layer;
  a.num_pages = geom->num_pages;
  a.page_size = geom->page_size;
  a.k = static_cast<const uint4 *>(k);
  a.v = static_cast<const uint4 *>(v);
  a.row_chunks = (int)(row / 8);
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.active = active;
  a.batch = batch;
  a.err = err_word;

  const int64_t warps = (int64_t)batch * 2;  // one per (row, K or V)
  int64_t blocks = (warps + APPEND_THREADS / 32 - 1) / (APPEND_THREADS / 32);
  if (blocks > 4096) blocks = 4096;
  if (launch_pdl(kv_append_kernel, dim3((unsigned)blocks), dim3(APPEND_THREADS), 0,
                 static_cast<cudaStream_t>(stream), a) != cudaSuccess)
    return PKV_ERR_CUDA;
  return launch_status();
}

extern "C" int pkv_kv_append_tokens(const pkv_cache_t *geom, void *cache, int layer, const void *k,
                                    const void *v, int total_tokens, const int32_t *qo_indptr,
                                    const int32_t *page_table, int max_pages,
                                    const int32_t *seq_lens, const int32_t *active, int batch,
                                    int32_t *err_word, void *stream) {
  using namespace pkv;
  int st = check_geometry(geom);
  if (st != PKV_OK) return st;
  if (!cache || !k || !v || !qo_indptr || !page_table || !seq_lens || !active)
    return PKV_ERR_INVALID_ARG;
  if (batch <= 0 || total_tokens <= 0 || max_pages <= 0 || layer < 0 ||
      layer >= geom->num_layers)
    return PKV_ERR_INVALID_ARG;
  const int64_t row = (int64_t)geom->num_kv_heads * geom->head_dim;
  if (row % 8 != 0) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(cache) || !aligned16(k) || !aligned16(v)) return PKV_ERR_INVALID_ARG;

  AppendTokArgs t;
  AppendArgs &a = t.base;
  a.cache = static_cast<uint4 *>(cache);
  a.slot_stride = row / 8;
  a.kv_stride = a.slot_stride * geom->page_size;
  a.page_stride = a.kv_stride * 2;
  a.layer_off = a.page_stride * (int64_t)geom->num_pages * layer;
  a.num_pages = geom->num_pages;
  a.page_size = geom->page_size;
  a.k = static_cast<const uint4 *>(k);
  a.v = static_cast<const uint4 *>(v);
  a.row_chunks = (int)(row / 8);
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.active = active;
  a.batch = batch;
  a.err = err_word;
  t.qo_indptr = qo_indptr;
  t.total_tokens = total_tokens;

  const int64_t warps = (int64_t)total_tokens * 2;  // one per (token, K or V)
  int64_t blocks = (warps + APPEND_THREADS / 32 - 1) / (APPEND_THREADS / 32);
  if (blocks > 8192) blocks = 8192;
  if (launch_pdl(kv_append_tokens_kernel, dim3((unsigned)blocks), dim3(APPEND_THREADS), 0,
                 static_cast<cudaStream_t>(stream), t) != cudaSuccess)
    return PKV_ERR_CUDA;
  return launch_status();
}
