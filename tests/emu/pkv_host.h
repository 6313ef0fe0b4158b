// Host stand-in for csrc/pkv_host.h in the CPU emulation test.
#pragma once
#include <cstddef>
namespace pkv {
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
}  // namespace pkv
