// Top-k selection over the logits: for every row, the column indices of its
// k largest finite logits (DeepSeek Sparse Attention keeps the top 2048 keys
// of each query). -inf (out of the row's window) is never selected; a row
// with fewer than k finite logits gets all of them and -1 in the remaining
// slots. Indices come out in no particular order; among equal values at the
// threshold any subset of the right size is taken.
//
// One CTA per row, radix select on an order-preserving 32-bit key of the
// value, 8 bits per digit from the top. Sweep 1 histograms the top digit and
// sweep 2 the second one among the elements matching it (per-warp
// sub-histograms in shared memory); each picks the digit where the count from
// the top reaches the number still to select. Sweep 3 writes the columns
// whose top 16 bits are above the threshold's and compacts the ones equal to
// it (the boundary bin, typically a few hundred) into shared memory, where
// the two low digits are resolved and the last columns picked. If the
// boundary bin does not fit, the low digits are resolved by further sweeps
// over the row instead. The row is read three times (five on the fallback);
// after the first it comes from L2.
#pragma once
#include <cstdint>

namespace dsa {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkCand = 3072;  // boundary-bin entries kept in shared memory

// Larger value -> larger key; -inf -> 0x007fffff, below every finite value.
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}
constexpr uint32_t kNegInfKey = 0x007fffffu;

template <bool BF16_IN>
__device__ __forceinline__ uint32_t load_key(const void* row, int j) {
  if constexpr (BF16_IN) {
    const uint32_t b = static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t*>(row) + j));
    return order_key(b << 16);
  } else {
    return order_key(__float_as_uint(__ldg(reinterpret_cast<const float*>(row) + j)));
  }
}

// Visits every column j < N of the row with f(j, key); four keys per load
// when the row start is 16-byte aligned (FP32) or 8-byte aligned (BF16).
template <bool BF16_IN, typename F>
__device__ __forceinline__ void for_each_key(const char* rp, int N, F&& f) {
  const int tid = threadIdx.x;
  const bool vec = (reinterpret_cast<uintptr_t>(rp) & (BF16_IN ? 7u : 15u)) == 0;
  const int n4 = vec ? N / 4 : 0;
  for (int q = tid; q < n4; q += kTopkThreads) {
    if constexpr (BF16_IN) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(rp) + q);
      f(4 * q, order_key(v.x << 16));
      f(4 * q + 1, order_key(v.x & 0xffff0000u));
      f(4 * q + 2, order_key(v.y << 16));
      f(4 * q + 3, order_key(v.y & 0xffff0000u));
    } else {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(rp) + q);
      f(4 * q, order_key(v.x));
      f(4 * q + 1, order_key(v.y));
      f(4 * q + 2, order_key(v.z));
      f(4 * q + 3, order_key(v.w));
    }
  }
  for (int j = 4 * n4 + tid; j < N; j += kTopkThreads) f(j, load_key<BF16_IN>(rp, j));
}

struct TopkShared {
  uint32_t hist[kTopkWarps][256];
  uint32_t total[256];
  uint32_t cand_key[kTopkCand];
  int32_t cand_idx[kTopkCand];
  uint32_t prefix, mask, need, finite, out, ties, ncand;
};

// Sum the per-warp histograms, then (warp 0) fix the digit at `shift` where
// the count from the top reaches sh.need: lane l owns digits 8l .. 8l+7 and a
// suffix sum over the lanes gives the count above each lane. Records the
// number of finite candidates in sh.finite when asked. Ends with a barrier.
__device__ __forceinline__ void topk_pick_digit(TopkShared& sh, int shift, bool count_finite) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __syncthreads();
  if (tid < 256) {
    uint32_t c = 0;
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) c += sh.hist[w][tid];
    sh.total[tid] = c;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t need = sh.need, prefix = sh.prefix, mask = sh.mask;
    uint32_t c[8], own = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c[i] = sh.total[8 * lane + i];
      own += c[i];
    }
    uint32_t suffix = own;  // this lane and the ones above
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_down_sync(0xffffffffu, suffix, o);
      if (lane + o < 32) suffix += v;
    }
    if (count_finite) {
      const uint32_t fin = __shfl_sync(0xffffffffu, suffix, 0);
      if (lane == 0) sh.finite = fin;
    }
    uint32_t above = suffix - own;
    if (above < need && need <= above + own) {
      int d = 8 * lane;
#pragma unroll
      for (int i = 7; i >= 0; --i) {
        if (above + c[i] >= need) {
          d = 8 * lane + i;
          break;
        }
        above += c[i];
      }
      sh.prefix = prefix | (static_cast<uint32_t>(d) << shift);
      sh.mask = mask | (255u << shift);
      sh.need = need - above;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ void topk_clear_hist(TopkShared& sh) {
  for (int i = threadIdx.x; i < kTopkWarps * 256; i += kTopkThreads) (&sh.hist[0][0])[i] = 0;
  __syncthreads();
}

template <bool BF16_IN>
__global__ void __launch_bounds__(kTopkThreads)
    topk_rows_kernel(const void* __restrict__ logits, int64_t row_stride, int N, int k,
                     int32_t* __restrict__ idx, int64_t idx_stride) {
  __shared__ TopkShared sh;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const char* rp = reinterpret_cast<const char*>(logits) + row * row_stride * (BF16_IN ? 2 : 4);
  int32_t* out = idx + row * idx_stride;
  if (tid == 0) {
    sh.prefix = 0;
    sh.mask = 0;
    sh.need = static_cast<uint32_t>(k);  // still to select at or below the fixed bits
    sh.finite = 0;
    sh.out = 0;
    sh.ties = 0;
    sh.ncand = 0;
  }

  // Sweeps 1 and 2: the top two digits.
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = 24 - 8 * pass;
    topk_clear_hist(sh);
    const uint32_t prefix = sh.prefix, mask = sh.mask;
    for_each_key<BF16_IN>(rp, N, [&](int, uint32_t key) {
      if (key > kNegInfKey && (key & mask) == prefix)
        atomicAdd(&sh.hist[warp][(key >> shift) & 255u], 1u);
    });
    topk_pick_digit(sh, shift, pass == 0);
    if (sh.finite <= static_cast<uint32_t>(k)) break;
  }

  if (sh.finite <= static_cast<uint32_t>(k)) {
    // every finite value is selected
    for_each_key<BF16_IN>(rp, N, [&](int j, uint32_t key) {
      if (key > kNegInfKey) out[atomicAdd(&sh.out, 1u)] = j;
    });
  } else {
    // Sweep 3: columns above the boundary bin are in; the bin is compacted.
    const uint32_t hi16 = sh.prefix >> 16;
    for_each_key<BF16_IN>(rp, N, [&](int j, uint32_t key) {
      if (key <= kNegInfKey) return;
      const uint32_t top = key >> 16;
      if (top > hi16) {
        out[atomicAdd(&sh.out, 1u)] = j;
      } else if (top == hi16) {
        const uint32_t pos = atomicAdd(&sh.ncand, 1u);
        if (pos < static_cast<uint32_t>(kTopkCand)) {
          sh.cand_key[pos] = key;
          sh.cand_idx[pos] = j;
        }
      }
    });
    __syncthreads();
    const uint32_t nc = sh.ncand;
    const bool in_smem = nc <= static_cast<uint32_t>(kTopkCand);
    // The two low digits, from the compacted bin or by sweeps over the row.
    for (int pass = 2; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      topk_clear_hist(sh);
      const uint32_t prefix = sh.prefix, mask = sh.mask;
      if (in_smem) {
        for (uint32_t c = tid; c < nc; c += kTopkThreads) {
          const uint32_t key = sh.cand_key[c];
          if ((key & mask) == prefix) atomicAdd(&sh.hist[warp][(key >> shift) & 255u], 1u);
        }
      } else {
        for_each_key<BF16_IN>(rp, N, [&](int, uint32_t key) {
          if (key > kNegInfKey && (key & mask) == prefix)
            atomicAdd(&sh.hist[warp][(key >> shift) & 255u], 1u);
        });
      }
      topk_pick_digit(sh, shift, false);
    }
    // The boundary bin's share: keys above the threshold, then enough ties.
    const uint32_t thr = sh.prefix, ties = sh.need;
    auto take = [&](int j, uint32_t key) {
      if ((key >> 16) != hi16) return;
      bool t = key > thr;
      if (key == thr) t = atomicAdd(&sh.ties, 1u) < ties;
      if (t) out[atomicAdd(&sh.out, 1u)] = j;
    };
    if (in_smem) {
      for (uint32_t c = tid; c < nc; c += kTopkThreads) take(sh.cand_idx[c], sh.cand_key[c]);
    } else {
      for_each_key<BF16_IN>(rp, N, [&](int j, uint32_t key) {
        if (key > kNegInfKey) take(j, key);
      });
    }
  }
  __syncthreads();
  for (int i = static_cast<int>(sh.out) + tid; i < k; i += kTopkThreads) out[i] = -1;
}

}  // namespace dsa
