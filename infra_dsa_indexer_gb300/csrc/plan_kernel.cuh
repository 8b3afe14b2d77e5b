// Row planning for irregular windows.
//
// The logits kernel computes a 4-row block over the union of its rows' key
// tiles. With consecutive rows and unrelated windows (workload: window start
// uniform in [0, N/2), length uniform in [0, N/2]) that union is ~2.4x the
// tiles the rows need. This kernel orders each batch's rows so that four
// consecutive positions have similar windows: rows are bucketed into strips of
// 1024 keys by window start, ordered within a strip by window end (ascending
// in even strips, descending in odd ones, so neighbouring strips meet), and
// empty rows go last. On that workload the blocks then cover 1.03x the tiles
// the rows need; for causal windows the order is the identity.
//
// One CTA per batch sorts 64-bit keys (strip, end, row) in shared memory with
// a bitonic network; S <= kPlanMaxRows.
#pragma once
#include <cstdint>

namespace dsa {

constexpr int kPlanMaxRows = 16384;  // 128 KB of keys in shared memory
constexpr int kPlanThreads = 1024;
constexpr int kStripShift = 10;      // strips of 1024 keys

__host__ __device__ inline int plan_pow2(int s) {
  int n = 1;
  while (n < s) n <<= 1;
  return n;
}

__global__ void __launch_bounds__(kPlanThreads, 1)
    plan_rows_kernel(const int32_t* __restrict__ ks, const int32_t* __restrict__ ke, int S, int N,
                     int32_t* __restrict__ perm) {
  extern __shared__ uint64_t keys[];
  const int b = blockIdx.x;
  const int n2 = plan_pow2(S);
  for (int i = threadIdx.x; i < n2; i += blockDim.x) {
    uint64_t key = ~0ull;  // padding sorts last
    if (i < S) {
      const int64_t row = static_cast<int64_t>(b) * S + i;
      const int lo = min(max(ks[row], 0), N);
      const int hi = min(max(ke[row], 0), N);
      uint64_t strip, end;
      if (lo < hi) {
        strip = static_cast<uint64_t>(lo >> kStripShift);
        end = static_cast<uint64_t>((strip & 1) ? N - hi : hi);
      } else {
        strip = (1ull << 19) - 1;  // empty rows after every strip
        end = 0;
      }
      key = (strip << 45) | (end << 21) | static_cast<uint64_t>(i);
    }
    keys[i] = key;
  }
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t a = keys[i], c = keys[ixj];
          const bool ascending = (i & k) == 0;
          if ((a > c) == ascending) {
            keys[i] = c;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < S; i += blockDim.x)
    perm[static_cast<int64_t>(b) * S + i] = static_cast<int32_t>(keys[i] & ((1u << 21) - 1));
}

}  // namespace dsa
