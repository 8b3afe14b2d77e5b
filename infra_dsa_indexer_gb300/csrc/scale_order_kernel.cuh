// Key scale words of MX keys rearranged, per 128-key tile, into the order in
// which the logits kernel copies them to tensor memory, so that its K
// producer moves a tile's 512 bytes with one bulk copy instead of 128
// four-byte copies (which sat on the MXFP8 tile loop: 4.3% of the call).
//
// Word 4l + c of tile t of batch b holds the scale word (four E8M0 bytes, one
// per 32 elements of D) of key 128t + 32c + l, zero past N: the 32 x 16-byte
// rows that tcgen05.cp.32x128b.warpx4 reads, row l = keys l, 32+l, 64+l, 96+l
// of the tile. Keys come from the dense [B, N] scale array, or through the
// block table of a paged cache.
#pragma once

#include <cstdint>

namespace dsa {

__global__ void scale_order_kernel(const uint32_t* __restrict__ k_sf, int N, int tiles,
                                   int64_t total_words, const int32_t* __restrict__ block_table,
                                   int64_t table_stride, int page_size, int num_pages,
                                   uint32_t* __restrict__ out) {
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < total_words;
       w += step) {
    const int64_t bt = w >> 7;  // (batch, tile)
    const int i = static_cast<int>(w & 127);
    const int64_t b = bt / tiles;
    const int t = static_cast<int>(bt - b * tiles);
    const int key = t * 128 + 32 * (i & 3) + (i >> 2);
    uint32_t v = 0u;
    if (key < N) {
      int64_t row = b * N + key;
      if (block_table != nullptr) {
        int page = __ldg(block_table + b * table_stride + key / page_size);
        page = page < 0 ? 0 : (page >= num_pages ? num_pages - 1 : page);
        row = static_cast<int64_t>(page) * page_size + key % page_size;
      }
      v = __ldg(k_sf + row);
    }
    out[w] = v;
  }
}

}  // namespace dsa
