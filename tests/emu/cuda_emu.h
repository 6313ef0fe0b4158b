// CPU emulation of the CUDA primitives the sampler kernels use, for running
// their CUDA source on the host in a test: one block at a time, every thread
// of the block a std::thread, __syncthreads a std::barrier over the block,
// warp shuffles / ballots / reductions a barrier-separated exchange over the
// warp's 32 threads (stricter than hardware: lanes never run in lockstep, so
// warp-synchronous assumptions show up as wrong results), atomics as GCC
// atomics.  Test infrastructure only.
#pragma once
#include <atomic>
#include <barrier>
#include <cmath>
#include <math.h>
#include <cstdint>
#include <cstring>
#include <cstdio>
#include <cstdlib>
#include <thread>
#include <vector>
#include <functional>

#define __device__
#define __global__
#define __host__
#define __forceinline__ inline
#define __noinline__ __attribute__((noinline))
#define __constant__
#define __shared__ static
#define __launch_bounds__(...)
#define __align__(n) alignas(n)
#define __restrict__

struct uint3_ { unsigned x = 0, y = 0, z = 0; };
struct dim3 { unsigned x = 1, y = 1, z = 1; dim3(unsigned a = 1, unsigned b = 1, unsigned c = 1) : x(a), y(b), z(c) {} };
inline thread_local uint3_ threadIdx;
inline uint3_ blockIdx;
inline dim3 blockDim, gridDim;

struct EmuWarp {
  std::barrier<> bar{32};
  uint64_t slot[32];
};
struct EmuBlock {
  std::barrier<> *bar = nullptr;
  EmuWarp *warps = nullptr;
};
inline EmuBlock g_block;

inline void __syncthreads() { g_block.bar->arrive_and_wait(); }
inline std::atomic<int> g_sync_or{0};
inline int __syncthreads_or(int pred) {
  if (pred) g_sync_or.store(1);
  g_block.bar->arrive_and_wait();
  const int r = g_sync_or.load();
  g_block.bar->arrive_and_wait();
  if (threadIdx.x == 0) g_sync_or.store(0);
  g_block.bar->arrive_and_wait();
  return r;
}
inline std::atomic<int> g_sync_and_miss{0};
inline int __syncthreads_and(int pred) {
  if (!pred) g_sync_and_miss.store(1);
  g_block.bar->arrive_and_wait();
  const int r = g_sync_and_miss.load() == 0;
  g_block.bar->arrive_and_wait();
  if (threadIdx.x == 0) g_sync_and_miss.store(0);
  g_block.bar->arrive_and_wait();
  return r;
}
inline EmuWarp &emu_warp() { return g_block.warps[threadIdx.x / 32]; }
inline void __syncwarp(unsigned = 0xffffffffu) { emu_warp().bar.arrive_and_wait(); }

template <class T> inline uint64_t emu_bits(T v) { uint64_t b = 0; std::memcpy(&b, &v, sizeof(T)); return b; }
template <class T> inline T emu_from(uint64_t b) { T v; std::memcpy(&v, &b, sizeof(T)); return v; }
template <class T> inline T emu_shfl_src(T v, int src) {
  EmuWarp &w = emu_warp();
  const int lane = threadIdx.x & 31;
  w.slot[lane] = emu_bits(v);
  w.bar.arrive_and_wait();
  const uint64_t r = w.slot[src & 31];
  w.bar.arrive_and_wait();
  return emu_from<T>(r);
}
template <class T> inline T __shfl_sync(unsigned, T v, int src) { return emu_shfl_src(v, src); }
template <class T> inline T __shfl_xor_sync(unsigned, T v, int m) { return emu_shfl_src(v, (int)(threadIdx.x & 31) ^ m); }
template <class T> inline T __shfl_up_sync(unsigned, T v, unsigned d) {
  const int lane = threadIdx.x & 31;
  const int src = lane - (int)d;
  T r = emu_shfl_src(v, src < 0 ? lane : src);
  return r;
}
inline unsigned __ballot_sync(unsigned, int pred) {
  EmuWarp &w = emu_warp();
  const int lane = threadIdx.x & 31;
  w.slot[lane] = pred ? 1 : 0;
  w.bar.arrive_and_wait();
  unsigned m = 0;
  for (int i = 0; i < 32; ++i) m |= (w.slot[i] ? 1u : 0u) << i;
  w.bar.arrive_and_wait();
  return m;
}
inline int __reduce_add_sync(unsigned, int v) {
  EmuWarp &w = emu_warp();
  const int lane = threadIdx.x & 31;
  w.slot[lane] = (uint64_t)(uint32_t)v;
  w.bar.arrive_and_wait();
  int s = 0;
  for (int i = 0; i < 32; ++i) s += (int)(uint32_t)w.slot[i];
  w.bar.arrive_and_wait();
  return s;
}
inline int __reduce_min_sync(unsigned, int v) {
  EmuWarp &w = emu_warp();
  const int lane = threadIdx.x & 31;
  w.slot[lane] = (uint64_t)(uint32_t)v;
  w.bar.arrive_and_wait();
  int m = (int)(uint32_t)w.slot[0];
  for (int i = 1; i < 32; ++i) m = (int)(uint32_t)w.slot[i] < m ? (int)(uint32_t)w.slot[i] : m;
  w.bar.arrive_and_wait();
  return m;
}
template <class T> inline T atomicAdd(T *p, T v) { return __atomic_fetch_add(p, v, __ATOMIC_SEQ_CST); }
template <class T> inline T atomicOr(T *p, T v) { return __atomic_fetch_or(p, v, __ATOMIC_SEQ_CST); }
template <class T> inline T atomicMin(T *p, T v) {
  T old = __atomic_load_n(p, __ATOMIC_SEQ_CST);
  while (v < old && !__atomic_compare_exchange_n(p, &old, v, false, __ATOMIC_SEQ_CST, __ATOMIC_SEQ_CST)) {
  }
  return old;
}

inline unsigned __float_as_uint(float f) { return emu_from<unsigned>(emu_bits(f)); }
inline float __uint_as_float(unsigned u) { return emu_from<float>((uint64_t)u); }
inline int __float_as_int(float f) { return emu_from<int>(emu_bits(f)); }
inline float __int_as_float(int i) { return emu_from<float>((uint64_t)(uint32_t)i); }
inline float __fadd_rn(float a, float b) { volatile float r = a + b; return r; }
inline float __fsub_rn(float a, float b) { volatile float r = a - b; return r; }
inline float __fmul_rn(float a, float b) { volatile float r = a * b; return r; }
inline float __fdiv_rn(float a, float b) { volatile float r = a / b; return r; }
inline float __ull2float_rn(unsigned long long u) { return (float)u; }
inline uint64_t __umul64hi(uint64_t a, uint64_t b) { return (uint64_t)(((unsigned __int128)a * b) >> 64); }
inline int __ffs(unsigned x) { return __builtin_ffs((int)x); }
inline int __popc(unsigned x) { return __builtin_popcount(x); }
inline int __clz(int x) { return x == 0 ? 32 : __builtin_clz((unsigned)x); }
inline long long clock64() { return 0; }
template <class T> inline T __ldg(const T *p) { return *p; }
template <class T> inline T __ldcg(const T *p) { return __atomic_load_n(p, __ATOMIC_SEQ_CST); }
inline void __threadfence() { std::atomic_thread_fence(std::memory_order_seq_cst); }
inline int min(int a, int b) { return a < b ? a : b; }
inline int max(int a, int b) { return a > b ? a : b; }
inline unsigned min(unsigned a, unsigned b) { return a < b ? a : b; }
inline unsigned max(unsigned a, unsigned b) { return a > b ? a : b; }
struct alignas(16) uint4 { unsigned x, y, z, w; };
struct alignas(16) ulonglong2 { unsigned long long x, y; };
inline uint4 make_uint4(unsigned x, unsigned y, unsigned z, unsigned w) { return {x, y, z, w}; }





// Shared memory starts undefined on the device: each block's static shared
// object is overwritten with a byte pattern first (EMU_SMEM_FILL, default
// 0xA5), so that a read of what the block did not write shows up.
inline void emu_poison_shared(void *p, size_t n) {
  if (threadIdx.x == 0) {
    const char *e = std::getenv("EMU_SMEM_FILL");
    const int v = e != nullptr ? (int)std::strtol(e, nullptr, 0) : 0xA5;
    std::memset(p, v, n);
  }
  g_block.bar->arrive_and_wait();
}

// run kernel(args) over grid with SB threads per block, one block at a time
template <class K, class A>
inline void emu_launch(K kern, dim3 grid, int threads, const A &a) {
  gridDim = grid;
  blockDim = dim3(threads);
  std::barrier<> bar(threads);
  std::vector<EmuWarp> warps(threads / 32);
  g_block.bar = &bar;
  g_block.warps = warps.data();
  for (unsigned by = 0; by < grid.y; ++by)
    for (unsigned bx = 0; bx < grid.x; ++bx) {
      blockIdx.x = bx; blockIdx.y = by; blockIdx.z = 0;
      std::vector<std::thread> ts;
      ts.reserve(threads);
      for (int t = 0; t < threads; ++t)
        ts.emplace_back([&, t] { threadIdx.x = t; threadIdx.y = 0; threadIdx.z = 0; kern(a); });
      for (auto &th : ts) th.join();
    }
}
