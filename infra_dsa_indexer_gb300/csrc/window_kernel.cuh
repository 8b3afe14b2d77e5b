// Per-row windows of sequences packed along the rows and keys of one batch
// (the THD / varlen layout of cuDNN-frontend pull request 416, "What": ragged
// sequences with absolute windows into the packed key axis and global key
// columns in the output).
//
// Sequence s owns query rows [cu_q[s], cu_q[s+1]) and keys [cu_k[s],
// cu_k[s+1]). Its query row r (0-based within the sequence) sees
//   [cu_k[s], cu_k[s] + clamp(n_k - n_q + r + 1, 0, n_k))   causal: the last
//                                                           row sees all n_k
//   [cu_k[s], cu_k[s+1])                                    otherwise
// with n_q, n_k the sequence's row and key counts. Rows at or past cu_q[num]
// get an empty window [0, 0).
#pragma once
#include <cstdint>

namespace dsa {

constexpr int kWindowThreads = 256;

__global__ void __launch_bounds__(kWindowThreads)
    thd_windows_kernel(const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k,
                       int num_seqs, int total_q, int causal, int32_t* __restrict__ ks,
                       int32_t* __restrict__ ke) {
  const int i = blockIdx.x * kWindowThreads + threadIdx.x;
  if (i >= total_q) return;
  if (i >= __ldg(cu_q + num_seqs)) {
    ks[i] = 0;
    ke[i] = 0;
    return;
  }
  // the sequence: the last s with cu_q[s] <= i (empty sequences have
  // cu_q[s] == cu_q[s+1] and are skipped by taking the last)
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu_q + mid) <= i) lo = mid;
    else hi = mid - 1;
  }
  const int q0 = __ldg(cu_q + lo), nq = __ldg(cu_q + lo + 1) - q0;
  const int k0 = __ldg(cu_k + lo), nk = __ldg(cu_k + lo + 1) - k0;
  int len = nk;
  if (causal) {
    len = nk - nq + (i - q0) + 1;
    len = len < 0 ? 0 : (len > nk ? nk : len);
  }
  ks[i] = k0;
  ke[i] = k0 + len;
}

}  // namespace dsa
