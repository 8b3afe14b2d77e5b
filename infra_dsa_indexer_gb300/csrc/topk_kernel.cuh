// Top-k selection over the logits: for every row, the column indices of its
// k largest finite logits (DeepSeek Sparse Attention keeps the top 2048 keys
// of each query). -inf (out of the row's window) is never selected; a row
// with fewer than k finite logits gets all of them and -1 in the remaining
// slots. Indices come out in no particular order; among equal values at the
// threshold any subset of the right size is taken.
//
// One CTA per row. Fast path: a sample of the row in shared memory sets a
// threshold a little below the expected k-th value, one sweep compacts the
// columns above it (k plus about three standard deviations of the sample's
// estimate), and the selection finishes in shared memory.
// Exact path (when the sample misjudges): radix select on an order-preserving
// 32-bit key of the value, 8 bits per digit from the top. Sweep 1 histograms the top digit and
// sweep 2 the second one among the elements matching it (one 256-bin
// histogram in shared memory); each picks the digit where the count from
// the top reaches the number still to select. Sweep 3 writes the columns
// whose top 16 bits are above the threshold's and compacts the ones equal to
// it (the boundary bin, typically a few hundred) into shared memory, where
// the two low digits are resolved and the last columns picked. If the
// boundary bin does not fit, the low digits are resolved by further sweeps
// over the row instead. The row is read three times (five on the fallback);
// after the first it comes from L2.
#pragma once
#include <cstdint>
#include <type_traits>

namespace dsa {

constexpr int kTopkThreads = 512;       // threads per CTA, four CTAs per SM
constexpr int kTopkThreadsFew = 1024;   // when the rows do not fill the GPU
constexpr int kTopkCand = 3840;  // candidate entries kept in shared memory

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
// The loads of kUnroll consecutive strides are issued before any key is
// visited, so each CTA keeps 32 KB of its row in flight.
template <int NT, bool BF16_IN, typename F>
__device__ __forceinline__ void for_each_key(const char* rp, int N, F&& f) {
  const int tid = threadIdx.x;
  const bool vec = (reinterpret_cast<uintptr_t>(rp) & (BF16_IN ? 7u : 15u)) == 0;
  const int n4 = vec ? N / 4 : 0;
  using V = typename std::conditional<BF16_IN, uint2, uint4>::type;
  constexpr int kUnroll = BF16_IN ? 8 : 4;
  const V* src = reinterpret_cast<const V*>(rp);
  auto visit = [&](int q, const V& v) {
    if constexpr (BF16_IN) {
      f(4 * q, order_key(v.x << 16));
      f(4 * q + 1, order_key(v.x & 0xffff0000u));
      f(4 * q + 2, order_key(v.y << 16));
      f(4 * q + 3, order_key(v.y & 0xffff0000u));
    } else {
      f(4 * q, order_key(v.x));
      f(4 * q + 1, order_key(v.y));
      f(4 * q + 2, order_key(v.z));
      f(4 * q + 3, order_key(v.w));
    }
  };
  int q = tid;
  for (; q + (kUnroll - 1) * NT < n4; q += kUnroll * NT) {
    V v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = __ldg(src + q + u * NT);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) visit(q + u * NT, v[u]);
  }
  for (; q < n4; q += NT) visit(q, __ldg(src + q));
  for (int j = 4 * n4 + tid; j < N; j += NT) f(j, load_key<BF16_IN>(rp, j));
}

struct TopkShared {
  uint32_t hist[256];
  uint32_t cand_key[kTopkCand];
  int32_t cand_idx[kTopkCand];
  uint32_t prefix, mask, need, finite, out, ties, ncand;
  uint32_t kmin, kmax;
};

// Warp 0 fixes the digit at `shift` where the histogram's count from the
// top reaches sh.need: lane l owns digits 8l .. 8l+7 and a suffix sum over
// the lanes gives the count above each lane. Records the number of finite
// candidates in sh.finite when asked. Ends with a barrier.
//
// One histogram for the whole block measured faster than per-warp copies
// (which spread the atomics but cost a summation and a larger clear each
// digit): the keys a digit counts are spread over its bins.
__device__ __forceinline__ void topk_pick_digit(TopkShared& sh, int shift, bool count_finite,
                                                uint32_t digit_mask = 255u) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __syncthreads();
  if (warp == 0) {
    const uint32_t need = sh.need, prefix = sh.prefix, mask = sh.mask;
    uint32_t c[8], own = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c[i] = sh.hist[8 * lane + i];
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
      sh.mask = mask | (digit_mask << shift);
      sh.need = need - above;
    }
  }
  __syncthreads();
}

template <int NT>
__device__ __forceinline__ void topk_clear_hist(TopkShared& sh) {
  for (int i = threadIdx.x; i < 256; i += NT) sh.hist[i] = 0;
  __syncthreads();
}

// Radix select of the sh.need-th largest among keys[0, n) in shared memory
// (0 marks an empty slot, below every finite key; sh.need must not exceed
// the non-zero keys): sh.prefix ends as its key, sh.need as the number of
// keys equal to it still to take. With max_digits, only that many 8-bit
// digits are resolved: sh.prefix then holds the key's leading bits with the
// rest zero, a lower bound of the key. The bits above the highest one where the
// non-zero keys differ are fixed at once, so the 8-bit digits start where the
// keys spread (the candidates of a row share their top bits, and a digit
// they all share would pile every lane's count onto one counter).
template <int NT>
__device__ __forceinline__ void topk_select_in_smem(TopkShared& sh, const uint32_t* keys,
                                                    uint32_t n, int max_digits = 4) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    sh.kmin = ~0u;
    sh.kmax = 0u;
  }
  __syncthreads();
  uint32_t mn = ~0u, mx = 0u;
  for (uint32_t c = tid; c < n; c += NT) {
    const uint32_t key = keys[c];
    if (key != 0u) {
      mn = min(mn, key);
      mx = max(mx, key);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if ((tid & 31) == 0) {
    atomicMin(&sh.kmin, mn);
    atomicMax(&sh.kmax, mx);
  }
  __syncthreads();
  const uint32_t kmin = sh.kmin, kmax = sh.kmax;
  // highest differing bit p (-1: all equal); bits above p are common
  const int p = kmin >= kmax ? -1 : 31 - __clz(kmin ^ kmax);
  const uint32_t common = p < 0 ? ~0u : (p >= 31 ? 0u : ~((2u << p) - 1u));
  __syncthreads();
  if (tid == 0) {
    sh.prefix = kmax & common;
    sh.mask = common;
  }
  int hi = p + 1;  // bits [0, hi) are still free
  for (int d = 0; hi > 0 && d < max_digits; ++d) {
    const int shift = hi > 8 ? hi - 8 : 0;
    const uint32_t width_mask = (1u << (hi - shift)) - 1u;
    topk_clear_hist<NT>(sh);
    const uint32_t prefix = sh.prefix, mask = sh.mask;
    for (uint32_t c = tid; c < n; c += NT) {
      const uint32_t key = keys[c];
      if (key != 0u && (key & mask) == prefix)
        atomicAdd(&sh.hist[(key >> shift) & width_mask], 1u);
    }
    topk_pick_digit(sh, shift, false, width_mask);
    hi = shift;
  }
  __syncthreads();
}

// Rows the selection reads, each a sequence of n (column, key) elements
// with random access by position e (key(e), col(e)) and a block-wide sweep
// (for_each(f): f(column, key) for every element).

// A dense logits row: element e is column e.
template <bool BF16_IN>
struct DenseRow {
  const char* rp;
  int n;
  __device__ __forceinline__ uint32_t key(int e) const { return load_key<BF16_IN>(rp, e); }
  __device__ __forceinline__ int col(int e) const { return e; }
  template <int NT, typename F>
  __device__ __forceinline__ void for_each(F&& f) const {
    for_each_key<NT, BF16_IN>(rp, n, f);
  }
};

// The fused top-k call's row: a compact FP32 sample row (element e < ns is
// column (e / 128) * 128 * sample_every + e % 128) followed by the kept-value
// slots of the filtered tiles, 32-slot group g with mask word mask[g]: slot
// 32 g + l holds a kept value iff bit l is set, for column
// tile(g / 4) * 128 + (g % 4) * 32 + l, where tile(r) is the r-th tile not
// sampled; unset slots are not elements (key 0).
struct MergeRow {
  const float* s;
  int ns;
  const float* kept;
  const uint32_t* mask;
  int ngroups;
  int sample_every;
  int n;
  __device__ __forceinline__ int sample_col(int e) const {
    return (e >> 7) * (128 * sample_every) + (e & 127);
  }
  __device__ __forceinline__ int kept_col(int g, int l) const {
    const int r = g >> 2;  // rank among the filtered tiles
    const int per = sample_every - 1;
    const int tile = (r / per) * sample_every + r % per + 1;
    return tile * 128 + (g & 3) * 32 + l;
  }
  // A group's kept values are packed at the front of its 32 slots in key
  // order: the value of mask bit l is at slot popc(mask & (2^l - 1)).
  __device__ __forceinline__ uint32_t key(int e) const {
    if (e < ns) return order_key(__float_as_uint(__ldg(s + e)));
    const int i = e - ns;
    const uint32_t m = __ldg(mask + (i >> 5));
    return (m >> (i & 31)) & 1u
               ? order_key(__float_as_uint(
                     __ldg(kept + (i & ~31) + __popc(m & ((1u << (i & 31)) - 1u)))))
               : 0u;
  }
  __device__ __forceinline__ int col(int e) const {
    return e < ns ? sample_col(e) : kept_col((e - ns) >> 5, (e - ns) & 31);
  }
  template <int NT, typename F>
  __device__ __forceinline__ void for_each(F&& f) const {
    for_each_key<NT, false>(reinterpret_cast<const char*>(s), ns,
                            [&](int e, uint32_t key) { f(sample_col(e), key); });
    // A warp takes 32 groups at a time: lane l reads mask word g0 + l; then,
    // eight groups at a time (eight independent loads in flight, within the
    // 32 registers of a thread at four CTAs per SM), every lane whose bit is
    // set in a group loads that key's packed slot (the group's first
    // sectors), then visits them.
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t below = (1u << lane) - 1u;
    for (int g0 = warp * 32; g0 < ngroups; g0 += NT) {
      const uint32_t mw = g0 + lane < ngroups ? __ldg(mask + g0 + lane) : 0u;
#pragma unroll
      for (int c = 0; c < 32; c += 8) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t m = __shfl_sync(0xffffffffu, mw, c + i);
          v[i] = (m >> lane) & 1u ? __ldg(kept + (g0 + c + i) * 32 + __popc(m & below)) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t m = __shfl_sync(0xffffffffu, mw, c + i);
          if ((m >> lane) & 1u) f(kept_col(g0 + c + i, lane), order_key(__float_as_uint(v[i])));
        }
      }
    }
  }
};

// The value of an order-preserving key.
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Where a selection puts its answer: the k column indices of the row
// (kth == nullptr), or only the k-th largest value (a lower bound of it, or
// -inf when the row has no more than k finite values) in *kth.
struct TopkOut {
  int32_t* idx;
  float* kth;
};

// Fast path (sample select). Runs of 8 consecutive elements spread over the
// row (in shared memory) give a threshold a little
// below the expected k-th largest value; one sweep compacts every element at
// or above it, and the exact selection runs on those in shared memory.
// Returns false, with nothing written, when the sample misjudged: fewer than
// k elements reach the threshold although it excluded finite values, or more
// elements than fit.
template <int NT, typename Src>
__device__ bool topk_sample_select(TopkShared& sh, const Src& src, int k, TopkOut o) {
  const int tid = threadIdx.x;
  const int N = src.n;
  constexpr int kRun = 8;
  // Sample size: enough runs that the k-th column's expected sample rank,
  // m = k * ns / N, is about 128 (spread ~9%), at least 512 keys and at
  // most the candidate buffer. A larger sample only lengthens the shared-
  // memory select; a smaller one sends more rows to the exact path.
  const int64_t want_runs = ((128LL * N + max(k, 1) - 1) / max(k, 1) + kRun - 1) / kRun;
  const int runs =
      static_cast<int>(want_runs < 64 ? 64 : (want_runs > kTopkCand / kRun ? kTopkCand / kRun
                                                                            : want_runs));
  const int step = N >= kRun * runs ? (N / runs) / kRun * kRun : kRun;
  if (tid == 0) {
    sh.ncand = 0;
    sh.prefix = 0;
    sh.mask = 0;
  }
  __syncthreads();
  uint32_t nfin_local = 0;
  for (int s = tid; s < runs * kRun; s += NT) {
    const int j = (s / kRun) * step + s % kRun;
    const uint32_t key = j < N ? src.key(j) : 0u;
    const bool fin = key > kNegInfKey;
    sh.cand_key[s] = fin ? key : 0u;  // 0 ranks below every finite key
    nfin_local += fin ? 1u : 0u;
  }
  const int ns = min(N, runs * step) / step * kRun + min(kRun, min(N, runs * step) % step);
  atomicAdd(&sh.ncand, nfin_local);
  __syncthreads();
  const uint32_t nfin = sh.ncand;
  // The sample rank m = k * ns / N is expected to have k columns of the row
  // at or above it; its count among the sample varies by about sqrt(m), so
  // the threshold goes to rank m + 3 sqrt(m) (+4), which leaves fewer than k
  // columns above it only rarely (the exact path then redoes the row).
  const float m = static_cast<float>(k) * static_cast<float>(ns) / static_cast<float>(N);
  const uint32_t r = static_cast<uint32_t>(ceilf(m + 3.f * sqrtf(m))) + 4u;
  uint32_t t_est = kNegInfKey + 1u;  // every finite value
  if (r <= nfin) {
    if (tid == 0) sh.need = r;
    // Two digits below the sample's common bits place the threshold within
    // 1/65536 of the sample's key range under its r-th largest key; the few
    // extra columns this admits cost nothing, and the exact selection below
    // needs no exact threshold.
    topk_select_in_smem<NT>(sh, sh.cand_key, runs * kRun, 2);
    t_est = max(sh.prefix, kNegInfKey + 1u);  // never admit -inf
  }
  __syncthreads();
  if (tid == 0) {
    sh.ncand = 0;
    sh.prefix = 0;
    sh.mask = 0;
    sh.need = static_cast<uint32_t>(k);
    sh.out = 0;
    sh.ties = 0;
  }
  __syncthreads();
  src.template for_each<NT>([&](int j, uint32_t key) {
    if (key < t_est) return;
    const uint32_t pos = atomicAdd(&sh.ncand, 1u);
    if (pos < static_cast<uint32_t>(kTopkCand)) {
      sh.cand_key[pos] = key;
      sh.cand_idx[pos] = j;
    }
  });
  __syncthreads();
  const uint32_t nc = sh.ncand;
  if (nc > static_cast<uint32_t>(kTopkCand)) return false;
  if (nc < static_cast<uint32_t>(k)) {
    // right only when the threshold let every finite value through
    if (t_est != kNegInfKey + 1u) return false;
    if (o.kth != nullptr) {
      if (tid == 0) *o.kth = __int_as_float(0xff800000);
      return true;
    }
    for (uint32_t c = tid; c < nc; c += NT) o.idx[c] = sh.cand_idx[c];
    for (int i = static_cast<int>(nc) + tid; i < k; i += NT) o.idx[i] = -1;
    return true;
  }
  topk_select_in_smem<NT>(sh, sh.cand_key, nc);
  const uint32_t thr = sh.prefix, ties = sh.need;
  if (o.kth != nullptr) {
    if (tid == 0) *o.kth = key_value(thr);
    return true;
  }
  for (uint32_t c = tid; c < nc; c += NT) {
    const uint32_t key = sh.cand_key[c];
    bool t = key > thr;
    if (key == thr) t = atomicAdd(&sh.ties, 1u) < ties;
    if (t) o.idx[atomicAdd(&sh.out, 1u)] = sh.cand_idx[c];
  }
  return true;
}

// The whole selection of one row by the CTA: the sample-select fast path,
// else an exact radix select by sweeps over the row.
template <int NT, typename Src>
__device__ void topk_row(TopkShared& sh, const Src& src, int k, TopkOut o) {
  const int tid = threadIdx.x;
  if (topk_sample_select<NT>(sh, src, k, o)) return;

  // Exact path: radix select by sweeps over the row.
  __syncthreads();
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
    topk_clear_hist<NT>(sh);
    const uint32_t prefix = sh.prefix, mask = sh.mask;
    src.template for_each<NT>([&](int, uint32_t key) {
      if (key > kNegInfKey && (key & mask) == prefix)
        atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
    });
    topk_pick_digit(sh, shift, pass == 0);
    if (sh.finite <= static_cast<uint32_t>(k)) break;
  }

  if (sh.finite <= static_cast<uint32_t>(k)) {
    if (o.kth != nullptr) {
      // no more than k finite values: no threshold excludes any of them
      if (tid == 0) *o.kth = __int_as_float(0xff800000);
      return;
    }
    // every finite value is selected
    src.template for_each<NT>([&](int j, uint32_t key) {
      if (key > kNegInfKey) o.idx[atomicAdd(&sh.out, 1u)] = j;
    });
  } else {
    // Sweep 3: columns above the boundary bin are in; the bin is compacted.
    const uint32_t hi16 = sh.prefix >> 16;
    const bool want_idx = o.kth == nullptr;
    src.template for_each<NT>([&](int j, uint32_t key) {
      if (key <= kNegInfKey) return;
      const uint32_t top = key >> 16;
      if (top > hi16) {
        if (want_idx) o.idx[atomicAdd(&sh.out, 1u)] = j;
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
      topk_clear_hist<NT>(sh);
      const uint32_t prefix = sh.prefix, mask = sh.mask;
      if (in_smem) {
        for (uint32_t c = tid; c < nc; c += NT) {
          const uint32_t key = sh.cand_key[c];
          if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
        }
      } else {
        src.template for_each<NT>([&](int, uint32_t key) {
          if (key > kNegInfKey && (key & mask) == prefix)
            atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
        });
      }
      topk_pick_digit(sh, shift, false);
    }
    // The boundary bin's share: keys above the threshold, then enough ties.
    const uint32_t thr = sh.prefix, ties = sh.need;
    if (!want_idx) {
      if (tid == 0) *o.kth = key_value(thr);
      return;
    }
    auto take = [&](int j, uint32_t key) {
      if ((key >> 16) != hi16) return;
      bool t = key > thr;
      if (key == thr) t = atomicAdd(&sh.ties, 1u) < ties;
      if (t) o.idx[atomicAdd(&sh.out, 1u)] = j;
    };
    if (in_smem) {
      for (uint32_t c = tid; c < nc; c += NT) take(sh.cand_idx[c], sh.cand_key[c]);
    } else {
      src.template for_each<NT>([&](int j, uint32_t key) {
        if (key > kNegInfKey) take(j, key);
      });
    }
  }
  __syncthreads();
  for (int i = static_cast<int>(sh.out) + tid; i < k; i += NT) o.idx[i] = -1;
}

// NT threads per CTA and 2048 / NT CTAs per SM (the register cap this
// implies costs a few spills). With many rows, 512 threads and four CTAs
// per SM: the shared-memory phases of one row overlap the sweeps of the
// others. With too few rows to fill the GPU (decode), 1024 threads per row
// shorten each row's sweeps and shared-memory passes instead.
//
// Launched as a programmatic dependent of the kernel before it on the stream
// (typically the logits kernel): its blocks may be placed while that kernel
// finishes, and wait here until it has completed and its writes are visible
// (a no-op when launched without the attribute).
template <int NT, bool BF16_IN>
__global__ void __launch_bounds__(NT, 2048 / NT)
    topk_rows_kernel(const void* __restrict__ logits, int64_t row_stride, int N, int k,
                     int32_t* __restrict__ idx, int64_t idx_stride) {
  __shared__ TopkShared sh;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t row = blockIdx.x;
  const DenseRow<BF16_IN> src{
      reinterpret_cast<const char*>(logits) + row * row_stride * (BF16_IN ? 2 : 4), N};
  topk_row<NT>(sh, src, k, TopkOut{idx + row * idx_stride, nullptr});
}

// Fused top-k, pass 2: the k-th largest value of each compact sample row
// (-inf if it holds no more than k finite values). k sample values of the
// row are logits of the row, so its k-th largest logit is at least this.
template <int NT>
__global__ void __launch_bounds__(NT, 2048 / NT)
    topk_threshold_kernel(const float* __restrict__ s, int64_t s_stride, int ns, int k,
                          float* __restrict__ thr) {
  __shared__ TopkShared sh;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // see topk_rows_kernel
  const int64_t row = blockIdx.x;
  const DenseRow<false> src{reinterpret_cast<const char*>(s + row * s_stride), ns};
  topk_row<NT>(sh, src, k, TopkOut{nullptr, thr + row});
}

// Fused top-k, pass 4: the k largest of a row's sample values and its kept
// candidates (every logit of the row at or above the threshold is in one
// of the two), as column indices.
template <int NT>
__global__ void __launch_bounds__(NT, 2048 / NT)
    topk_merge_kernel(const float* __restrict__ s, int64_t s_stride, int ns,
                      const float* __restrict__ kept, int64_t kept_stride,
                      const uint32_t* __restrict__ mask, int64_t mask_stride, int sample_every,
                      int k, int32_t* __restrict__ idx, int64_t idx_stride) {
  __shared__ TopkShared sh;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // see topk_rows_kernel
  const int64_t row = blockIdx.x;
  const int ngroups = static_cast<int>(mask_stride);
  const MergeRow src{s + row * s_stride, ns, kept + row * kept_stride, mask + row * mask_stride,
                     ngroups, sample_every, ns + 32 * ngroups};
  topk_row<NT>(sh, src, k, TopkOut{idx + row * idx_stride, nullptr});
}

}  // namespace dsa
