// fastdiv.h -- division of 32-bit unsigned integers by a divisor fixed at launch time, as one
// multiply-high, a subtraction, an add and two shifts (Granlund and Montgomery, "Division by
// Invariant Integers using Multiplication", PLDI 1994, section 4, the round-up method with a
// 33-bit multiplier 2^32 + m).  Plain C++: the host computes the constants, the kernel divides,
// and a host test checks the result against the built-in division.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define SPECV_HD __host__ __device__ __forceinline__
#else
#define SPECV_HD inline
#endif

namespace specv {

struct FastDiv {
  uint32_t d;    // divisor (>= 1)
  uint32_t m;    // low 32 bits of the multiplier
  uint32_t sh1;  // min(l, 1)
  uint32_t sh2;  // max(l - 1, 0), where l = ceil(log2(d))
};

// Constants for divisor d >= 1: l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1.
inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  uint32_t l = 0;
  while (l < 32 && (uint64_t(1) << l) < d) ++l;
  f.m = (uint32_t)(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
  f.sh1 = l < 1 ? l : 1;
  f.sh2 = l > 1 ? l - 1 : 0;
  return f;
}

SPECV_HD uint32_t mulhi_u32(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
  return __umulhi(a, b);
#else
  return (uint32_t)(((uint64_t)a * b) >> 32);
#endif
}

// n / d for every 32-bit n.
SPECV_HD uint32_t fdiv(uint32_t n, const FastDiv& f) {
  const uint32_t t1 = mulhi_u32(f.m, n);
  return (t1 + ((n - t1) >> f.sh1)) >> f.sh2;
}

}  // namespace specv
