// pkv_api.cu -- library-wide helpers of the C ABI declared in include/pkv.h.
#include "pkv.h"

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
