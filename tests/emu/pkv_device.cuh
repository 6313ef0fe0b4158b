// Host stand-in for csrc/pkv_device.cuh, used only by the CPU emulation test
// of the sampler kernels (tests/test_sampler_emulated.py): the CUDA
// primitives come from cuda_emu.h, error reporting is an atomic OR.
#pragma once
#include "cuda_emu.h"
#include "pkv.h"
namespace pkv {
constexpr unsigned FULL_MASK = 0xffffffffu;
inline void report(int32_t *err, int bits) {
  if (err != nullptr) atomicOr(err, (int32_t)bits);
}
// one grid at a time here: the programmatic-launch hooks have nothing to do
inline void pdl_wait() {}
inline void pdl_trigger() {}
// the SFU's log2 (an approximation there; exact enough here)
inline float lg2_approx(float x) { return std::log2(x); }
}  // namespace pkv
