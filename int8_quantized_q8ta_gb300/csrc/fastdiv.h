// fastdiv.h -- division of 32-bit unsigned integers by a divisor fixed for
// a launch, by one multiply-high and two shifts: the method of Granlund and
// Montgomery, "Division by Invariant Integers using Multiplication" (PLDI
// 1994), Figure 4.1.  For d >= 2, with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, the quotient of any 32-bit n is
// (t + ((n - t) >> 1)) >> (l - 1), t = umulhi(m, n); d = 1 is m = 0 with both
// shifts 0.  Plain C++ on the host (make_fastdiv, fast_div_host); the
// device form uses __umulhi.  No CUDA header is needed to include it.
#pragma once

#include <cstdint>

namespace q8 {

struct FastDiv {
  uint32_t d, m, s1, s2;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f{d, 0u, 0u, 0u};
  if (d <= 1) {
    f.d = 1;
    return f;
  }
  uint32_t l = 0;
  while ((uint64_t{1} << l) < d) ++l;
  f.m = static_cast<uint32_t>(((uint64_t{1} << 32) * ((uint64_t{1} << l) - d)) / d + 1);
  f.s1 = 1;
  f.s2 = l - 1;
  return f;
}

// The same quotient on the host: the multiply-high in 64-bit arithmetic.
inline uint32_t fast_div_host(uint32_t n, const FastDiv& f) {
  const uint32_t t = static_cast<uint32_t>((static_cast<uint64_t>(f.m) * n) >> 32);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
  const uint32_t t = __umulhi(f.m, n);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

// q = n / f.d, r = n % f.d
__device__ __forceinline__ void fast_divmod(uint32_t n, const FastDiv& f, uint32_t& q, uint32_t& r) {
  q = fast_div(n, f);
  r = n - q * f.d;
}
#endif

}  // namespace q8
