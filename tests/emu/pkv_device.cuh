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
// asynchronous copies: plain copies here, with the hardware's alignment rule
// (both addresses aligned to the copy's size) checked
inline void emu_cp_async(void *dst, const void *src, size_t n) {
  if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) % n != 0) {
    std::fprintf(stderr, "misaligned cp.async of %zu bytes: dst %p src %p\n", n, dst, src);
    std::abort();
  }
  std::memcpy(dst, src, n);
}
inline void cp_async4(void *dst, const void *src) { emu_cp_async(dst, src, 4); }
inline void cp_async8(void *dst, const void *src) { emu_cp_async(dst, src, 8); }
inline void cp_async16(void *dst, const void *src) { emu_cp_async(dst, src, 16); }
inline void cp_async_wait_all() {}
// mbarriers and bulk copies: the copy is done when issued, so a barrier's
// phase is complete by the time anyone waits on it
inline void mbar_init(uint64_t *, uint32_t) {}
inline void fence_barrier_init() {}
inline void mbar_arrive_expect_tx(uint64_t *, uint32_t) {}
inline void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *) {
  if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | bytes) % 16 != 0) {
    std::fprintf(stderr, "misaligned bulk copy of %u bytes: dst %p src %p\n", bytes, dst, src);
    std::abort();
  }
  std::memcpy(dst, src, bytes);
}
inline bool mbar_wait(uint64_t *, uint32_t, uint64_t = 0) { return true; }
inline void __threadfence_block() { std::atomic_thread_fence(std::memory_order_seq_cst); }
// packed fp32 pairs: .x in the low half of a 64-bit word; every operation
// is the scalar IEEE one on each half
typedef unsigned long long f32x2;
inline f32x2 pack2(float a, float b) {
  uint32_t x, y;
  std::memcpy(&x, &a, 4);
  std::memcpy(&y, &b, 4);
  return (f32x2)x | ((f32x2)y << 32);
}
struct float2 { float x, y; };
inline float2 unpack2(f32x2 v) {
  const uint32_t x = (uint32_t)v, y = (uint32_t)(v >> 32);
  float2 r;
  std::memcpy(&r.x, &x, 4);
  std::memcpy(&r.y, &y, 4);
  return r;
}
inline f32x2 ffma2(f32x2 a, f32x2 b, f32x2 c) {
  const float2 A = unpack2(a), B = unpack2(b), C = unpack2(c);
  return pack2(std::fmaf(A.x, B.x, C.x), std::fmaf(A.y, B.y, C.y));
}
inline f32x2 fadd2(f32x2 a, f32x2 b) {
  const float2 A = unpack2(a), B = unpack2(b);
  return pack2(__fadd_rn(A.x, B.x), __fadd_rn(A.y, B.y));
}
inline f32x2 fsub2(f32x2 a, f32x2 b) {
  const float2 A = unpack2(a), B = unpack2(b);
  return pack2(__fsub_rn(A.x, B.x), __fsub_rn(A.y, B.y));
}
inline f32x2 fmul2(f32x2 a, f32x2 b) {
  const float2 A = unpack2(a), B = unpack2(b);
  return pack2(__fmul_rn(A.x, B.x), __fmul_rn(A.y, B.y));
}
// the SFU's exp2 (an approximation there; exact enough here)
inline float fast_exp2(float x) { return std::exp2(x); }
// the SFU's log2 (an approximation there; exact enough here)
inline float lg2_approx(float x) { return std::log2(x); }
}  // namespace pkv
