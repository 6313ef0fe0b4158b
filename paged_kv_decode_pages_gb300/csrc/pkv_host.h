// pkv_host.h -- host-side argument checks shared by the C-ABI entry points.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

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

// Status of the launches just made on this thread; does not synchronise.
inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace pkv
