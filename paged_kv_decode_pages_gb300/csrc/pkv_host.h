// pkv_host.h -- host-side argument checks shared by the C-ABI entry points.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "pkv.h"

namespace pkv {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int check_geometry(const pkv_cache_t *g) {
  if (g == nullptr) return PKV_ERR_INVALID_ARG;
  if (g->num_layers <= 0 || g->num_pages <= 0 || g->page_size <= 0 || g->num_kv_heads <= 0 ||
      g->head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

// The CUDA runtime error behind this thread's latest PKV_ERR_CUDA from
// launch_status() (pkv_last_cuda_error reads it).
void record_cuda_error(cudaError_t e);

// Status of the launches just made on this thread; does not synchronise.
inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return PKV_OK;
  record_cuda_error(e);
  return PKV_ERR_CUDA;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launch with programmatic stream serialization: the kernel may be scheduled
// while its predecessor on the stream is still running; it must call
// pdl_wait() before touching anything the predecessor may write.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace pkv
