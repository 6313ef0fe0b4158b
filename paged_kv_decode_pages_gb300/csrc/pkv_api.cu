// pkv_api.cu -- library-wide helpers of the C ABI declared in include/pkv.h.
#include "pkv_device.cuh"
#include "pkv_host.h"

extern "C" const char *pkv_version(void) { return "pkv 0.1.0 sm_103a"; }

extern "C" const char *pkv_error_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_CUDA: return "CUDA launch error";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

extern "C" int pkv_num_dev_error_bits(void) { return 7; }

namespace pkv {
static thread_local int g_last_cuda_error = 0;
void record_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }
}  // namespace pkv

extern "C" int pkv_last_cuda_error(void) {
  if (pkv::g_last_cuda_error != 0) return pkv::g_last_cuda_error;
  // a launch that failed before its status was read leaves its error pending
  return static_cast<int>(cudaPeekAtLastError());
}

extern "C" const char *pkv_cuda_error_name(int code) {
  return cudaGetErrorName(static_cast<cudaError_t>(code));
}

namespace pkv {

// one thread block waits, through the kernels' own bounded wait, on an
// mbarrier that nothing arrives on
__global__ void selftest_wait_kernel(unsigned long long limit_ns, int32_t *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (!__all_sync(FULL_MASK, mbar_wait_spin(&bar, 0u, limit_ns)) && threadIdx.x == 0)
    report(err, PKV_DEV_ERR_TIMEOUT);
}

}  // namespace pkv

extern "C" int pkv_selftest_wait_timeout(unsigned long long limit_ns, int32_t *err_word,
                                         void *stream) {
  if (err_word == nullptr || limit_ns == 0 || limit_ns > 1000000000ull) return PKV_ERR_INVALID_ARG;
  pkv::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, err_word);
  return pkv::launch_status();
}
