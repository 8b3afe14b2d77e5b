// Row planning for irregular windows.
//
// The logits kernel computes a 4-row block over the union of its rows' key
// tiles. With consecutive rows and unrelated windows (workload: window start
// uniform in [0, N/2), length uniform in [0, N/2]) that union is ~2.4x the
// tiles the rows need. This kernel orders each batch's rows so that four
// consecutive positions have similar windows: rows are binned by window
// start (strips of 1024 keys) and, within a strip, by window end (buckets of
// 128 keys, ascending in even strips and descending in odd ones, so
// neighbouring strips meet); empty rows go last. On that workload the blocks
// then cover ~1.03x the tiles the rows need; for causal windows rows keep
// their order up to swaps inside a bin.
//
// One CTA per batch does a counting sort in shared memory: a histogram of
// the bins, an exclusive scan, and a scatter. The order inside a bin follows
// the atomics and may differ between calls; the logits do not depend on the
// row order (each row is computed the same way in any block).
#pragma once
#include <cstdint>

namespace dsa {

constexpr int kPlanThreads = 1024;
constexpr int kPlanMaxBins = 49152;  // 192 KB of counters in shared memory
constexpr int kStripShift = 10;      // strips of 1024 keys
constexpr int kEndShift = 7;         // end buckets of 128 keys (one key tile)
constexpr int kPlanSmemBytes = (kPlanMaxBins + 32) * static_cast<int>(sizeof(int));

struct PlanGeometry {
  int sshift, eshift, ebn, nbins;  // nbins includes the last bin, for empty rows
};

// Bin sizes for N keys: the finest strips/buckets (at least 1024 / 128 keys)
// whose product fits the counters.
__device__ __forceinline__ PlanGeometry plan_geometry(int N) {
  PlanGeometry g;
  g.sshift = kStripShift;
  while (((N - 1) >> g.sshift) + 1 > 4096) ++g.sshift;
  const int strips = ((N - 1) >> g.sshift) + 1;
  g.eshift = kEndShift;
  while (strips * ((N >> g.eshift) + 1) + 1 > kPlanMaxBins) ++g.eshift;
  g.ebn = (N >> g.eshift) + 1;
  g.nbins = strips * g.ebn + 1;
  return g;
}

__device__ __forceinline__ int plan_bin(const PlanGeometry& g, int lo, int hi) {
  if (lo >= hi) return g.nbins - 1;
  const int strip = lo >> g.sshift;
  const int e = hi >> g.eshift;
  return strip * g.ebn + ((strip & 1) ? g.ebn - 1 - e : e);
}

__global__ void __launch_bounds__(kPlanThreads, 1)
    plan_rows_kernel(const int32_t* __restrict__ ks, const int32_t* __restrict__ ke, int S, int N,
                     int32_t* __restrict__ perm) {
  extern __shared__ int hist[];  // [kPlanMaxBins] counters, then 32 warp sums
  int* wsum = hist + kPlanMaxBins;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const PlanGeometry g = plan_geometry(N);
  const int64_t base = static_cast<int64_t>(b) * S;
  auto bin_of = [&](int i) {
    const int lo = min(max(__ldg(ks + base + i), 0), N);
    const int hi = min(max(__ldg(ke + base + i), 0), N);
    return plan_bin(g, lo, hi);
  };

  for (int i = tid; i < g.nbins; i += kPlanThreads) hist[i] = 0;
  __syncthreads();
  for (int i = tid; i < S; i += kPlanThreads) atomicAdd(&hist[bin_of(i)], 1);
  __syncthreads();

  // Exclusive scan of the counters in place: each thread a contiguous chunk,
  // the chunk sums scanned across the block.
  const int chunk = (g.nbins + kPlanThreads - 1) / kPlanThreads;
  const int c0 = min(g.nbins, tid * chunk), c1 = min(g.nbins, c0 + chunk);
  int sum = 0;
  for (int i = c0; i < c1; ++i) sum += hist[i];
  int x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int v = wsum[lane];  // kPlanThreads / 32 == 32 warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    wsum[lane] = v;
  }
  __syncthreads();
  int run = x - sum + (warp > 0 ? wsum[warp - 1] : 0);
  for (int i = c0; i < c1; ++i) {
    const int c = hist[i];
    hist[i] = run;
    run += c;
  }
  __syncthreads();

  for (int i = tid; i < S; i += kPlanThreads) {
    const int pos = atomicAdd(&hist[bin_of(i)], 1);
    perm[base + pos] = i;
  }
}

}  // namespace dsa
