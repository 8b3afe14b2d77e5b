// Division of a key index by the page size of a paged key cache, with one
// multiply-high and one shift instead of an integer division.
//
// For a divisor d >= 2 and a numerator n < 2^31 (every key index and every
// row of a cache is below 2^31), let l = ceil(log2 d) and m = ceil(2^(31+l) / d).
// Then floor(n / d) = floor(n * m / 2^(31+l)): writing m = 2^(31+l)/d + e with
// 0 <= e < 1, the product is n/d + n*e / 2^(31+l), and n*e / 2^(31+l) <
// 2^-l <= 1/d, which cannot carry n/d past the next integer (its fractional
// part is at most (d-1)/d). m < 2^32 because d > 2^(l-1). This is the
// round-up method of T. Granlund and P. L. Montgomery, "Division by invariant
// integers using multiplication" (PLDI 1994), for 31-bit numerators.
// The high word of the 64-bit product n*m is n*m / 2^32, so the quotient is
// that word shifted right by l - 1.
#pragma once
#include <cstdint>

namespace dsa {

struct PageDiv {
  uint32_t magic;  // m
  int32_t shift;   // l - 1
};

// d in [2, 2^31].
inline PageDiv page_div_make(uint32_t d) {
  int l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  const uint64_t m = ((uint64_t(1) << (31 + l)) + d - 1) / d;
  return PageDiv{static_cast<uint32_t>(m), l - 1};
}

// floor(n / d) for n < 2^31, with (magic, shift) = page_div_make(d).
#ifdef __CUDACC__
__host__ __device__
#endif
inline uint32_t page_div(uint32_t n, uint32_t magic, int32_t shift) {
#ifdef __CUDA_ARCH__
  return __umulhi(n, magic) >> shift;
#else
  return static_cast<uint32_t>((static_cast<uint64_t>(n) * magic) >> 32) >> shift;
#endif
}

}  // namespace dsa
