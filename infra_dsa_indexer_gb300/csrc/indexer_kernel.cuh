// Lightning-indexer MQA-logits forward, one persistent warp-specialised
// kernel for sm_103a.
//
//   out[b,i,j] = sum_h w[b,i,h] * ReLU(sm_scale * q[b,i,h,:] . k[b,j,:])  (ks <= j < ke)
//   out[b,i,j] = -inf                                                     (otherwise)
//
// The operation is the "fp8_fp4_mqa_logits" call of DeepGEMM pull request 435
// ("Improve SM100 MX MQA logits clean-output performance", standalone
// performance reproducer) and the BF16 indexer forward of cuDNN-frontend pull
// request 416 ("DSA indexer forward: add a lean SM100 fast path ...",
// sections "What" and "Precision / determinism").
//
// Work decomposition (own design; the pages' kernels are prior art):
//  * row-block = 4 query rows of one batch (consecutive, or consecutive in
//    the row planner's order; the last block of a batch may have fewer) =
//    4 x 64 heads = 256 (row, head) pairs; key tile = 128 keys, contiguous
//    per batch or read through a page table (PAGED).
//  * One tcgen05 MMA group per (row-block, key tile) with swapped operands:
//    A = key tile (M = 128 keys), B = the row-block's Q (N = 256 (row,head)),
//    K = D = 128. The FP32 accumulator lands in TMEM with one key per lane and
//    one (row, head) per column, so the head reduction sum_h w*ReLU(s*x) is a
//    per-thread loop over columns: no shuffles, no shared-memory reduction.
//  * Kinds: BF16 kind::f16; E4M3 kind::f8f6f4; MXFP8 kind::mxf8f6f4 and MXFP4
//    kind::mxf4, block-scaled with one E8M0 scale per 32 elements of D held in
//    TMEM next to the accumulator.
//  * A unit of work is (row-block, chunk of its key tiles). Units are handed
//    out through a global atomic counter, longest row-blocks first (for causal
//    windows the highest row index), so the persistent grid balances itself.
//
// Roles (one CTA per SM; 4 role warps + 8 or 16 epilogue warps):
//  warp 0       K-tile TMA producer (lane 0; paged keys: the first of the
//               tile's two 64-key boxes, each inside one page); for MX
//               formats the tile's key scale factors come along, one 512-byte
//               bulk copy of words a pre-pass put in the order the TMEM copy
//               reads (without library scratch, all 32 lanes copy them key by
//               key)
//  warp 1       TMEM allocator + MMA issuer (one lane)
//  warp 2       unit scheduler: claims a unit and fetches its windows, head
//               weights and (MX) Q scale factors into registers; when the Q
//               half of a slot frees it starts the TMA of the unit's Q block
//               (and stages the Q scale factors), when the epilogue half
//               frees it stages the weights in shared memory as FP32 and the
//               windows, one unit ahead of the MMA; with paged keys it also
//               copies the unit's first 32 block-table entries for the
//               producers and the epilogue
//  warp 3       paged keys: the second 64-key box of every tile (one thread
//               issuing TMA boxes of 8 KB tops out near 4.4 TB/s of HBM per
//               GPU; two issuing warps near 6.9), else idle
//  warps 4..    epilogue, R = 1 or 2 query rows per warp (a per-format
//               choice): warp w reads TMEM lanes 32*(w%4)..+31 (the
//               sub-partition it may access) of rows R*((w-4)/4) .. +R-1; it
//               loads its rows' accumulator columns, hands the buffer back to
//               the MMA warp, then does the ReLU.w head sums, the masked FP32
//               (or BF16) stores and the -inf fill outside the block's tiles. R = 2
//               (8 warps, 168 registers each) halves the per-tile overhead
//               (waits, stores, loop) and suits BF16, where the MMA is long,
//               and the MX formats, whose single accumulator serialises MMA
//               and epilogue anyway; R = 1 (16 warps) hides the epilogue's
//               latency better for E4M3, whose short MMA is double-buffered.
//               Paged E4M3 keys: two groups of 8 warps take alternate tiles
//               and each warp reduces two rows, one after the other, so one
//               group's loads and scale lookups overlap the other's sums.
// Pipelines (mbarriers): unit slots x2 (unit info + Q block + W [+ Q scales]),
// key-tile ring (kStages) [+ key scales], TMEM accumulators: two 256-column
// buffers, so the MMA of tile t+1 overlaps the epilogue of tile t, or one for
// the MX formats (their scale factors need TMEM too: two slots each).
#pragma once
#include <cuda.h>
#include <cstdint>

#include "page_div.h"
#include "ptx.cuh"

namespace dsa {

constexpr int kKeysPerTile = 128;  // MMA M
constexpr int kRowsPerBlock = 4;
constexpr int kHeads = 64;
constexpr int kBlockN = kRowsPerBlock * kHeads;  // MMA N = 256
constexpr int kHeadDim = 128;                    // MMA K per tile
constexpr int kEpiWarp0 = 4;
constexpr uint32_t kTmemCols = 512;
constexpr int kStepBytes = 32;                   // bytes of K per MMA instruction
constexpr uint32_t kSfaCol = 256;                // MX: key scale factors, 2 slots x 4 columns
constexpr uint32_t kSfbCol = 264;                // MX: Q scale factors, 2 slots x 8 columns
constexpr int kSfaBytes = kKeysPerTile * 4;      // one 32-bit word (4 E8M0) per key
constexpr int kSfbBytes = kBlockN * 4;           // one word per (row, head)

enum : int { kFmtBF16 = 0, kFmtE4M3 = 1, kFmtMXFP8 = 2, kFmtMXFP4 = 3 };
enum : int { kErrTimeout = 8, kErrAlign = 4 };

// What a launch computes (the fused top-k call runs the last two):
//  kModeLogits  every key tile; the logits go to `out` (the indexer call)
//  kModeSample  key tiles t with t % kSampleEvery == 0; their logits go to a
//               compact row of ceil(tiles / kSampleEvery) * 128 columns
//               (column (t / kSampleEvery) * 128 + j % 128), -inf outside
//               the window and past N
//  kModeFilter  the other key tiles; only in-window logits >= the row's
//               threshold thr[row] are kept. Key j of filtered tile t keeps
//               its value at slot rank(t) * 128 + j % 128 of the row's kept
//               values (rank(t): position of t among the filtered tiles),
//               and 32-key group g = rank(t) * 4 + (j % 128) / 32 has a mask
//               word (bit j % 32 set: kept) in the row's masks
enum : int { kModeLogits = 0, kModeSample = 1, kModeFilter = 2 };
constexpr int kSampleEvery = 4;

template <int MODE>
__device__ __forceinline__ bool tile_in_mode(int t) {
  if constexpr (MODE == kModeSample) return t % kSampleEvery == 0;
  else if constexpr (MODE == kModeFilter) return t % kSampleEvery != 0;
  else return true;
}
// First tile >= t that the mode computes.
template <int MODE>
__device__ __forceinline__ int first_tile(int t) {
  if constexpr (MODE == kModeSample) return (t + kSampleEvery - 1) / kSampleEvery * kSampleEvery;
  else if constexpr (MODE == kModeFilter) return t % kSampleEvery == 0 ? t + 1 : t;
  else return t;
}
template <int MODE>
__device__ __forceinline__ int next_tile(int t) {
  return first_tile<MODE>(t + 1);
}

struct UnitInfo {
  int32_t stop;
  int32_t b;
  int32_t row[4];    // flattened row ids b*S + i of the block's rows; -1: no such row
  int32_t c0, c1;    // key tiles [c0, c1) computed by this unit
  int32_t t0, t1;    // key tiles [t0, t1) covered by the whole row-block
  int32_t flags;     // bit 0: fill [0, t0*128) with -inf; bit 1: fill [t1*128, N)
  int32_t lo[4];     // clamped window per row
  int32_t hi[4];
};

// What the K producer and the MMA issuer need of a unit, published with its
// Q block (the rest of UnitInfo and the weights are the epilogue's).
struct QInfo {
  int32_t stop;
  int32_t b;
  int32_t c0, c1;
};

struct KernelParams {
  CUtensorMap tmap_q;  // [B*S*H rows, D] view of Q
  CUtensorMap tmap_k;  // [B, N, D] view of K, or [pages * page_size, D] of a paged cache
  const uint8_t* q_sf;
  const uint8_t* k_sf;
  // MX formats: the key scale words in tensor-memory copy order, 512 bytes per
  // (batch, 128-key tile) (scale_order_kernel); unused with SF_KEYS.
  const uint8_t* k_sf_tiles;
  const float* k_scales;
  const void* w;
  const int32_t* ks;
  const int32_t* ke;
  const int32_t* perm;  // [B,S] row order within each batch, or null (identity)
  // Paged keys (null: contiguous [B, N] keys): key j of batch b is row
  // j % page_size of page block_table[b * table_stride + j / page_size] of
  // the cache; key scales (k_sf, k_scales) follow the same rows.
  const int32_t* block_table;
  int32_t page_size;     // multiple of 64
  uint32_t page_magic;   // page_div_make(page_size): key / page_size without a division
  int32_t page_shift;
  int32_t table_stride;
  int32_t num_pages;     // page numbers are clamped to [0, num_pages)
  void* out;         // FP32, or BF16 when out_bf16; the compact sample rows
                     // (kModeSample) or the (value, column) candidates (kModeFilter)
  int32_t* scratch;  // [0] unit counter, [1] finished CTAs, [2] error word
  int64_t out_row_stride;  // elements (kModeFilter: candidate slots per row)
  const float* thr;        // kModeFilter: per-row threshold
  uint32_t* mask;          // kModeFilter: per-row group masks (zeroed before)
  int64_t mask_row_stride; // kModeFilter: mask words per row
  int32_t B, S, N;
  int32_t w_bf16;
  int32_t out_bf16;  // selects the OUT_BF16 instantiation
  int32_t clean;
  int32_t num_units;
  int32_t nchunk;
  int32_t blocks_per_batch;  // ceil(S / rows per block); the last block may be partial
  float sm_scale;
  uint64_t timeout_ns;
};

// Per-format constants. kRowBytes: bytes of one D=128 row of Q or K; the
// operands are K-major with a swizzle of kSwizzleBytes (TMA writes the same
// pattern), kPanels column panels of kSwizzleBytes each.
template <int FMT>
struct Traits;

template <>
struct Traits<kFmtBF16> {
  static constexpr int kRowBytes = kHeadDim * 2;
  static constexpr int kSwizzleBytes = 128;
  static constexpr int kTmaElemBytes = 2;
  static constexpr int kStages = 3;
  static constexpr uint32_t kIdesc = instr_desc(1, 1, kKeysPerTile, kBlockN);  // BF16 x BF16
  static constexpr int kKind = 0;
  static constexpr int kRowsPerWarp = 2;
  static constexpr bool kMX = false;
  static constexpr int kSfIdStep = 0;
  static constexpr bool kReluAllAdd = true;  // packed-add ReLU on every head pair (RowAcc)
};

template <>
struct Traits<kFmtE4M3> {
  static constexpr int kRowBytes = kHeadDim;
  static constexpr int kSwizzleBytes = 128;
  static constexpr int kTmaElemBytes = 1;
  static constexpr int kStages = 8;
  static constexpr uint32_t kIdesc = instr_desc(0, 0, kKeysPerTile, kBlockN);  // E4M3 x E4M3
  static constexpr int kKind = 1;
  static constexpr int kRowsPerWarp = 1;
  static constexpr bool kMX = false;
  static constexpr int kSfIdStep = 0;
  static constexpr bool kReluAllAdd = false;  // packed-add ReLU on every head pair (RowAcc)
};

template <>
struct Traits<kFmtMXFP8> {
  static constexpr int kRowBytes = kHeadDim;
  static constexpr int kSwizzleBytes = 128;
  static constexpr int kTmaElemBytes = 1;
  static constexpr int kStages = 8;
  // E4M3 x E4M3, UE8M0 scales, one per 32 elements: MMA step kk (K = 32) uses
  // scale byte kk of each row's 32-bit scale word.
  static constexpr uint32_t kIdesc = instr_desc_bs(0, 0, kKeysPerTile, kBlockN, 0, 0);
  static constexpr int kKind = 2;
  static constexpr int kRowsPerWarp = 2;
  static constexpr bool kMX = true;
  static constexpr int kSfIdStep = 1;
  static constexpr bool kReluAllAdd = true;  // packed-add ReLU on every head pair (RowAcc)
};

template <>
struct Traits<kFmtMXFP4> {
  static constexpr int kRowBytes = kHeadDim / 2;  // two E2M1 per byte
  static constexpr int kSwizzleBytes = 64;
  static constexpr int kTmaElemBytes = 1;           // the tensor map walks bytes
  static constexpr int kStages = 12;
  // E2M1 x E2M1, UE8M0 scales: MMA step kk (K = 64) uses scale bytes 2kk, 2kk+1.
  static constexpr uint32_t kIdesc = instr_desc_bs(1, 1, kKeysPerTile, kBlockN, 0, 0);
  static constexpr int kKind = 3;
  static constexpr int kRowsPerWarp = 2;
  static constexpr bool kMX = true;
  static constexpr int kSfIdStep = 2;
  static constexpr bool kReluAllAdd = true;  // packed-add ReLU on every head pair (RowAcc)
};

// RB: query rows per block, kRowsPerBlock, or 2 for batches of at most two
// rows (decode with one or two new tokens), where a four-row block would
// leave half of every MMA and of the epilogue warps without a row. With
// RB = 2 the MMA is N = 128 into four 128-column accumulators and the
// epilogue warps form two groups that take alternate tiles (BF16 and E4M3;
// the MX formats keep one accumulator and RB = 4).
template <int FMT, int RB = kRowsPerBlock>
struct Layout {
  using T = Traits<FMT>;
  static_assert(RB == kRowsPerBlock || (RB == 2 && !T::kMX), "rows per block");
  static constexpr int kNumEpiWarps = 4 * kRowsPerBlock / T::kRowsPerWarp;
  static constexpr int kThreads = (kEpiWarp0 + kNumEpiWarps) * 32;
  static constexpr int kBlockNR = RB * kHeads;                    // MMA N
  static constexpr int kGroups = kRowsPerBlock / RB;              // epilogue warp groups
  static constexpr int kAccBufs = T::kMX ? 1 : 2 * kGroups;       // accumulators of kBlockNR columns
  // The instruction descriptor with its N field (bits [17,23), N >> 3) set to kBlockNR.
  static constexpr uint32_t kIdesc = (T::kIdesc & ~(0x3Fu << 17)) | ((kBlockNR >> 3) << 17);
  static constexpr int kPanels = T::kRowBytes / T::kSwizzleBytes;
  static constexpr int kSteps = T::kRowBytes / kStepBytes;           // MMAs per tile
  static constexpr int kStepsPerPanel = T::kSwizzleBytes / kStepBytes;
  static constexpr int kAtomBytes = 8 * T::kSwizzleBytes;            // 8-row swizzle atom
  static constexpr int kKPanelBytes = kKeysPerTile * T::kSwizzleBytes;
  static constexpr int kQPanelBytes = kBlockNR * T::kSwizzleBytes;
  static constexpr int kKTileBytes = kKPanelBytes * kPanels;
  static constexpr int kQBlockBytes = kQPanelBytes * kPanels;
  static constexpr int kWBytes = RB * kHeads * 4;  // FP32 weights of a block
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + 2 * kQBlockBytes;
  static constexpr int kWOff = kKOff + T::kStages * kKTileBytes;
  static constexpr int kSfaOff = kWOff + 2 * kWBytes;
  static constexpr int kSfbOff = kSfaOff + (T::kMX ? T::kStages * kSfaBytes : 0);
  static constexpr int kInfoOff = kSfbOff + (T::kMX ? 2 * kSfbBytes : 0);
  static constexpr int kQInfoOff = kInfoOff + 2 * (int)sizeof(UnitInfo);
  static constexpr int kPagesOff = kQInfoOff + 2 * (int)sizeof(QInfo);
  static constexpr int kBarOff = kPagesOff + 4 * 32 * 4;  // paged: 32 table entries x 4
  static constexpr int kNumBars =
      2 + 2 + 2 * T::kStages + 2 * kAccBufs + (T::kMX ? T::kStages : 0) + 1 + 2 + 2;
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
  static constexpr int kBytes = kMiscOff + 16;
  static_assert(kBytes <= 232448, "shared memory budget");
};

__device__ __forceinline__ int clampi(int v, int lo, int hi) {
  return v < lo ? lo : (v > hi ? hi : v);
}

// Page of key (or cache row) j of a paged cache: j / page_size (j >= 0).
__device__ __forceinline__ int page_index(const KernelParams& p, int j) {
  return static_cast<int>(page_div(static_cast<uint32_t>(j), p.page_magic, p.page_shift));
}

__device__ __forceinline__ void raise_error(int32_t* scratch, volatile int* abort_flag, int code) {
  *abort_flag = 1;
  atomicExch(scratch + 2, code);
}

// Write -inf to columns [a, b) of one output row (FP32, or BF16 0xff80);
// the 128 threads of the four warps sharing `row` cover 128 consecutive
// columns per step.
__device__ __forceinline__ void fill_neg_inf(char* row, int a, int b, int tid128, bool bf16) {
  if (bf16) {
    for (int j = a + tid128; j < b; j += 128) st_cs_b16(row + 2 * static_cast<int64_t>(j), 0xff80);
  } else {
    const float ninf = __int_as_float(0xff800000);
    float* rowf = reinterpret_cast<float*>(row);
    for (int j = a + tid128; j < b; j += 128) __stcs(rowf + j, ninf);
  }
}

// sum_h w[h] * R(x[h]) over the 64 heads of a row, R(x) = max(x, 0) (NEG:
// min(x, 0)), taken four heads at a time and multiply-accumulated pairwise
// with packed FP32x2 FMAs. The ReLU of a pair is either two max on the ALU
// pipe, or one packed add x + |x| = 2 max(x, 0) on the FMA pipe (the packed
// add takes |x| as an operand modifier: one instruction for two heads).
// ALL_ADD uses the packed add for every pair; otherwise half the pairs use
// max, which balances the two pipes where the epilogue is the bottleneck.
// Doubled sums are halved at the end (exact). NEG is used only where the MMA
// cannot negate its A operand; it takes the scalar min / x - |x| forms.
template <bool NEG, bool ALL_ADD>
struct RowAcc {
  float2 m0, m1, d0, d1;
  __device__ __forceinline__ void zero() { m0 = m1 = d0 = d1 = make_float2(0.f, 0.f); }
  __device__ __forceinline__ void step(int g, float4 w, float x0, float x1, float x2, float x3) {
    float2 rm, rd;
    if constexpr (NEG) {
      rm = make_float2(fminf(x0, 0.f), fminf(x1, 0.f));
      rd = make_float2(x2 - fabsf(x2), x3 - fabsf(x3));
    } else {
      if constexpr (ALL_ADD)
        rm = __fadd2_rn(make_float2(x0, x1), make_float2(fabsf(x0), fabsf(x1)));
      else
        rm = make_float2(fmaxf(x0, 0.f), fmaxf(x1, 0.f));
      rd = __fadd2_rn(make_float2(x2, x3), make_float2(fabsf(x2), fabsf(x3)));
    }
    if (g & 1) {
      m1 = __ffma2_rn(make_float2(w.x, w.y), rm, m1);
      d1 = __ffma2_rn(make_float2(w.z, w.w), rd, d1);
    } else {
      m0 = __ffma2_rn(make_float2(w.x, w.y), rm, m0);
      d0 = __ffma2_rn(make_float2(w.z, w.w), rd, d0);
    }
  }
  __device__ __forceinline__ float total() const {
    const float sm = (m0.x + m0.y) + (m1.x + m1.y);
    const float sd = (d0.x + d0.y) + (d1.x + d1.y);
    if constexpr (ALL_ADD && !NEG) return 0.5f * (sm + sd);
    return fmaf(sd, 0.5f, sm);
  }
};

// Head groups [G0, G1) (4 heads each) of R rows at once: v[r] holds row r's
// 64 accumulator columns, w + r*64 its 64 FP32 weights in shared memory.
// Rows are interleaved for ILP.
template <int G0, int G1, int R, bool NEG, bool ALL_ADD>
__device__ __forceinline__ void head_steps(RowAcc<NEG, ALL_ADD> (&a)[R], const uint32_t (&v)[R][64],
                                           const float* w) {
#pragma unroll
  for (int g = G0; g < G1; ++g) {
#pragma unroll
    for (int r = 0; r < R; ++r)
      a[r].step(g, reinterpret_cast<const float4*>(w + r * kHeads)[g], __uint_as_float(v[r][4 * g]),
                __uint_as_float(v[r][4 * g + 1]), __uint_as_float(v[r][4 * g + 2]),
                __uint_as_float(v[r][4 * g + 3]));
  }
}

template <int KIND>
__device__ __forceinline__ void mma_step(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate, uint32_t sfa,
                                         uint32_t sfb) {
  if constexpr (KIND == 2) {
    tc_mma_mxf8f6f4(d_tmem, a_desc, b_desc, idesc, sfa, sfb, accumulate);
  } else if constexpr (KIND == 3) {
    tc_mma_mxf4(d_tmem, a_desc, b_desc, idesc, sfa, sfb, accumulate);
  } else {
    tc_mma<KIND>(d_tmem, a_desc, b_desc, idesc, accumulate);
  }
}

// NEG_EPI: the epilogue applies a negative sm_scale itself (MXFP4, whose MMA
// kind has no negate bit); every other case negates the MMA's A operand.
// OUT_BF16: the logits are stored as BF16 (round to nearest even).
// PAGED: the keys (and key scales) are read through the page table.
// MODE: kModeLogits, or one of the two passes of the fused top-k call.
// RB: rows per block (Layout).
// SF_KEYS (MX formats): the K producer copies each key's scale word itself
// (128 four-byte copies per tile, counted on their own barrier) instead of
// one bulk copy of the tile's words put in order beforehand; for calls
// without library scratch. A compile-time choice: as a run-time flag in the
// producer and MMA issuer loops it cost the MXFP8 kernel the whole 4% the
// bulk copy gains.
template <int FMT, bool NEG_EPI, bool OUT_BF16, bool PAGED, int MODE = kModeLogits,
          int RB = kRowsPerBlock, bool SF_KEYS = false>
__global__ void __launch_bounds__(Layout<FMT, RB>::kThreads, 1)
    indexer_logits_kernel(const __grid_constant__ KernelParams p) {
  static_assert(MODE == kModeLogits || (!OUT_BF16 && !PAGED), "fused top-k: FP32, contiguous keys");
  static_assert(RB == kRowsPerBlock || MODE == kModeLogits, "fused top-k: four-row blocks");
  static_assert(!SF_KEYS || (Traits<FMT>::kMX && !PAGED && MODE == kModeLogits),
                "per-key scale copies: contiguous MX logits only");
  using T = Traits<FMT>;
  using L = Layout<FMT, RB>;
  constexpr int kNumEpiWarps = L::kNumEpiWarps;
  constexpr int kAccBufs = L::kAccBufs;
  constexpr int R = T::kRowsPerWarp;
  // Row sets a warp reduces one after the other (each of R rows): two for
  // paged E4M3 four-row blocks, whose epilogue also makes the two dependent
  // loads of each key's page and scale. There the 16 warps form two groups
  // that take alternate tiles, each group with its own accumulator, so the
  // TMEM loads and scale lookups of one group overlap the other's sums
  // (measured: 8% faster on 64- and 256-key pages; on contiguous keys and
  // for BF16 the same arrangement was 1-5% slower).
  constexpr int kSeq = (FMT == kFmtE4M3 && PAGED && RB == kRowsPerBlock) ? 2 : 1;
  constexpr int kGroups = L::kGroups * kSeq;         // epilogue warp groups
  constexpr int kGroupWarps = kNumEpiWarps / kGroups;
  extern __shared__ __align__(1024) uint8_t smem[];

  uint8_t* qbuf = smem + L::kQOff;
  uint8_t* kbuf = smem + L::kKOff;
  uint8_t* wbuf = smem + L::kWOff;
  uint8_t* sfa_s = smem + L::kSfaOff;  // [kStages][128 keys x 4 bytes], TMEM-copy order
  uint8_t* sfb_s = smem + L::kSfbOff;  // [2 slots][256 rows x 4 bytes], TMEM-copy order
  UnitInfo* info = reinterpret_cast<UnitInfo*>(smem + L::kInfoOff);
  QInfo* qinfo = reinterpret_cast<QInfo*>(smem + L::kQInfoOff);
  // Paged keys: the first 32 block-table entries of each slot's unit, copied
  // by the scheduler for the K producer ([slot]) and the epilogue ([2 + slot]).
  int32_t* unit_pages = reinterpret_cast<int32_t*>(smem + L::kPagesOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  // A unit slot has two halves: the Q half (Q block, MX Q scales, QInfo;
  // q_full / q_empty), read by the K producer and the MMA issuer and
  // released by the MMA's commit, and the epilogue half (UnitInfo, weights;
  // unit_full / unit_empty), released by the epilogue warps. The Q half of
  // a slot is thus refilled as soon as the MMAs of its previous unit are
  // done, a tile or two before the epilogue is.
  uint64_t* unit_full = bars;
  uint64_t* unit_empty = bars + 2;
  uint64_t* k_full = bars + 4;
  uint64_t* k_empty = k_full + T::kStages;
  uint64_t* acc_full = k_empty + T::kStages;
  uint64_t* acc_empty = acc_full + kAccBufs;
  uint64_t* sf_full = acc_empty + kAccBufs;  // MX only
  uint64_t* drain = sf_full + (T::kMX ? T::kStages : 0);  // MMA issuer, after an abort
  uint64_t* q_full = drain + 1;
  uint64_t* q_empty = q_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    if ((smem_u32(smem) & 1023u) != 0) {
      // The swizzle atoms need a 1024-byte aligned base.
      atomicExch(p.scratch + 2, kErrAlign);
    }
    *abort_flag = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&unit_full[s], 1);                // the scheduler's arrive
      mbar_init(&unit_empty[s], kNumEpiWarps);    // epilogue warps
      mbar_init(&q_full[s], 1);                   // the scheduler's arrive + the Q TMA bytes
      mbar_init(&q_empty[s], 1);                  // the MMA issuer's commit
    }
    for (int s = 0; s < kAccBufs; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], kGroupWarps);  // the warps of the group that drains it
    }
    for (int s = 0; s < T::kStages; ++s) {
      mbar_init(&k_full[s], PAGED ? 2 : 1);  // paged: one arrive per producer warp
      mbar_init(&k_empty[s], 1);
      if constexpr (T::kMX) mbar_init(&sf_full[s], 32);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool misaligned = (smem_u32(smem) & 1023u) != 0;

  if (misaligned) {
    // nothing: the error word says why
  } else if (warp == 2) {
    // ---------------------------------------------------------- unit scheduler
    // A unit is claimed and its rows, windows, weights and (MX) Q scale
    // words are fetched into registers; once the Q half of its slot is free,
    // lane 0 writes the QInfo and starts the Q TMA and all lanes store the
    // scale words; once the epilogue half is free, lane 0 writes the unit
    // info and all lanes store the weights (FP32). Claiming and fetching take
    // several microseconds (a contended atomic, then dependent global
    // loads). With grouped rows (one more dependent load, the row order;
    // many short units) the next unit is claimed as soon as a slot frees
    // and fetched right after the current one is published, so that work
    // overlaps the units in flight; otherwise a unit is claimed only once
    // its slot is free, which keeps the tail of the persistent grid short.
    if (lane == 0) prefetch_tmap(&p.tmap_q);
    const uint64_t pol_first = policy_evict_first();  // Q block: read once per unit
    struct Prep {
      int u, chunk, blk, b;
      int grow[kRowsPerBlock];
      UnitInfo in;      // lane 0 only: the info the slot gets
      float4 w[2];      // this lane's part of the block's FP32 head weights
      int32_t pg;       // paged keys: table entry `lane` of the unit's first page on
      uint32_t sf[kBlockN / 32];  // MX: this lane's Q scale words
    };
    // grow[i] for a lane-dependent i, without indexing the array at run time
    // (which would move it to local memory).
    auto pick = [](const int (&g)[kRowsPerBlock], int i) {
      return i == 0 ? g[0] : i == 1 ? g[1] : i == 2 ? g[2] : g[3];
    };
    // Fetch everything unit u needs, into registers.
    auto prepare = [&](int u, Prep& q) {
      q.u = u;
      if (u >= p.num_units) return;
      // Units in order: row-blocks from the last (longest causal window) to
      // the first, batches interleaved, chunks of one row-block adjacent.
      const int order = u / p.nchunk;
      q.chunk = u - order * p.nchunk;
      q.blk = p.blocks_per_batch - 1 - order / p.B;
      q.b = order % p.B;
      // The block's rows: positions RB*blk .. RB*blk+RB-1 of the batch's row
      // order. Positions past S (a partial last block) read the batch's last
      // row in that order, so every address stays valid; the row gets an
      // empty window and is never stored. With RB = 2, rows 2 and 3 of the
      // unit info are absent and their addresses are those of row 0.
#pragma unroll
      for (int r = 0; r < kRowsPerBlock; ++r) {
        const int pos = min(q.blk * RB + (r < RB ? r : 0), p.S - 1);
        q.grow[r] = q.b * p.S + (p.perm != nullptr ? __ldg(p.perm + q.b * p.S + pos) : pos);
      }
      if (lane == 0) {
        int lo_all = p.N, hi_all = 0;
#pragma unroll
        for (int r = 0; r < kRowsPerBlock; ++r) {
          const bool exists = r < RB && q.blk * RB + r < p.S;
          const int lo = exists ? clampi(__ldg(p.ks + q.grow[r]), 0, p.N) : 0;
          const int hi = exists ? clampi(__ldg(p.ke + q.grow[r]), 0, p.N) : 0;
          q.in.row[r] = exists ? q.grow[r] : -1;
          q.in.lo[r] = lo;
          q.in.hi[r] = hi;
          if (lo < hi) {
            lo_all = min(lo_all, lo);
            hi_all = max(hi_all, hi);
          }
        }
        int t0 = 0, t1 = 0;
        if (lo_all < hi_all) {
          t0 = lo_all / kKeysPerTile;
          t1 = (hi_all + kKeysPerTile - 1) / kKeysPerTile;
        }
        const int len = (t1 - t0 + p.nchunk - 1) / p.nchunk;
        q.in.stop = 0;
        q.in.b = q.b;
        q.in.c0 = min(t1, t0 + q.chunk * len);
        q.in.c1 = min(t1, q.in.c0 + len);
        q.in.t0 = t0;
        q.in.t1 = t1;
        q.in.flags = (q.chunk == 0 ? 1 : 0) | (q.chunk == p.nchunk - 1 ? 2 : 0);
      }
      if constexpr (PAGED) {
        // The unit's first 32 table entries, loaded with the weights: the K
        // producer and the epilogue start the unit without waiting for the
        // table.
        const int c0 = __shfl_sync(0xffffffffu, q.in.c0, 0);
        const int c1 = __shfl_sync(0xffffffffu, q.in.c1, 0);
        const int e = page_index(p, c0 * kKeysPerTile) + lane;
        const int n_e = page_index(p, p.N - 1) + 1;
        q.pg = c0 < c1 && e < n_e
                   ? __ldg(p.block_table + static_cast<int64_t>(q.b) * p.table_stride + e)
                   : 0;
      }
      if (p.w_bf16) {
        // lane l: 8 weights = 16 bytes, row l/8, heads 8*(l%8).. (rows past
        // RB: row 0 again, not stored)
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p.w) +
                                static_cast<int64_t>(pick(q.grow, RB == kRowsPerBlock
                                                                      ? lane >> 3
                                                                      : (lane >> 3) % RB)) *
                                    (kHeads / 8) +
                                (lane & 7));
        q.w[0] = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                             __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u));
        q.w[1] = make_float4(__uint_as_float(raw.z << 16), __uint_as_float(raw.z & 0xffff0000u),
                             __uint_as_float(raw.w << 16), __uint_as_float(raw.w & 0xffff0000u));
      } else {
        // float4 f = lane + 32i: row f/16, heads 4*(f%16)..
        const float4* src = reinterpret_cast<const float4*>(p.w);
#pragma unroll
        for (int i = 0; i < RB / 2; ++i) {
          const int f = lane + 32 * i;
          q.w[i] = __ldg(src + static_cast<int64_t>(pick(q.grow, f >> 4)) * (kHeads / 4) + (f & 15));
        }
      }
      if constexpr (T::kMX) {
        // (row, head) m = 32c + lane = 64r + h: the word of row grow[r], head
        // h, with r = c / 2 (lane < 32).
#pragma unroll
        for (int c = 0; c < kBlockN / 32; ++c) {
          const int m = 32 * c + lane;
          q.sf[c] = __ldg(reinterpret_cast<const uint32_t*>(p.q_sf) +
                          static_cast<int64_t>(q.grow[c >> 1]) * kHeads + (m & 63));
        }
      }
    };
    const bool ahead = p.perm != nullptr;
    int u_next = 0;
    Prep cur;
    if (ahead) {
      if (lane == 0) u_next = atomicAdd(p.scratch + 0, 1);
      prepare(__shfl_sync(0xffffffffu, u_next, 0), cur);
    }
    // Waits for a slot half; on expiry, lets the Q loads still in flight
    // (units [first, last)) land before the CTA exits.
    auto wait_half = [&](uint64_t* bar, uint32_t it, uint32_t first, uint32_t last) {
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(&bar[it & 1], ((it >> 1) & 1) ^ 1, abort_flag, p.timeout_ns);
        if (!ok) {
          raise_error(p.scratch, abort_flag, kErrTimeout);
          for (uint32_t j = first; j < last; ++j)
            mbar_wait_drain(&q_full[j & 1], (j >> 1) & 1, p.timeout_ns);
        }
      }
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    for (uint32_t it = 0;; ++it) {
      const int slot = it & 1;
      // Q half: free once the MMAs of unit it-2 are done.
      if (!wait_half(q_empty, it, it > 2 ? it - 2 : 0, it)) break;
      if (!ahead) {
        if (lane == 0) u_next = atomicAdd(p.scratch + 0, 1);
        prepare(__shfl_sync(0xffffffffu, u_next, 0), cur);
      }
      QInfo& qi = qinfo[slot];
      UnitInfo& in = info[slot];
      if (cur.u >= p.num_units) {
        if (lane == 0) {
          qi.stop = 1;
          mbar_arrive(&q_full[slot]);
        }
        if (!wait_half(unit_empty, it, it > 1 ? it - 1 : 0, it)) break;
        if (lane == 0) {
          in.stop = 1;
          mbar_arrive(&unit_full[slot]);
        }
        break;
      }
      // The next claim; its result is first needed after this unit is out.
      if (ahead && lane == 0) u_next = atomicAdd(p.scratch + 0, 1);
      if (lane == 0) {
        qi.stop = 0;
        qi.b = cur.in.b;
        qi.c0 = cur.in.c0;
        qi.c1 = cur.in.c1;
        if (cur.in.c1 > cur.in.c0) {
          mbar_expect_tx(&q_full[slot], L::kQBlockBytes);
          // One 64-head box per row and panel; row r lands at rows 64r.. of
          // the block (a whole number of swizzle atoms).
          uint8_t* qdst = qbuf + slot * L::kQBlockBytes;
#pragma unroll
          for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int pnl = 0; pnl < L::kPanels; ++pnl)
              tma_load_2d(qdst + pnl * L::kQPanelBytes + r * kHeads * T::kSwizzleBytes,
                          &p.tmap_q, &q_full[slot], pnl * (T::kSwizzleBytes / T::kTmaElemBytes),
                          cur.grow[r] * kHeads, pol_first);
        }
      }
      if constexpr (T::kMX) {
        // Q scale word of (row, head) m = 32c + lane goes to TMEM lane m % 32,
        // column m / 32: in shared memory, chunk m / 128 (one TMEM copy
        // each), row m % 32 (16 bytes), word (m % 128) / 32.
        uint8_t* dst = sfb_s + slot * kSfbBytes;
#pragma unroll
        for (int c = 0; c < kBlockN / 32; ++c) {
          const int m = 32 * c + lane;
          *reinterpret_cast<uint32_t*>(dst + (m >> 7) * 512 + 16 * lane + 4 * (c & 3)) = cur.sf[c];
        }
      }
      if constexpr (PAGED) unit_pages[slot * 32 + lane] = cur.pg;
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[slot]);
      // Epilogue half: free once the epilogue is done with unit it-2.
      if (!wait_half(unit_empty, it, it > 1 ? it - 1 : 0, it + 1)) break;
      if (lane == 0) in = cur.in;
      if constexpr (PAGED) unit_pages[(2 + slot) * 32 + lane] = cur.pg;
      // Head weights of the RB rows as FP32, row-major RB x 64.
      float4* wdst = reinterpret_cast<float4*>(wbuf + slot * L::kWBytes);
      if (p.w_bf16) {
        if (RB == kRowsPerBlock || lane < 8 * RB) {
          wdst[2 * lane] = cur.w[0];
          wdst[2 * lane + 1] = cur.w[1];
        }
      } else {
#pragma unroll
        for (int i = 0; i < RB / 2; ++i) wdst[lane + 32 * i] = cur.w[i];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&unit_full[slot]);
      if (ahead) prepare(__shfl_sync(0xffffffffu, u_next, 0), cur);
    }
  } else if (PAGED ? (warp == 0 || warp == 3) : (warp == 0 && (T::kMX || lane == 0))) {
    // (Written as a compile-time choice: the form "warp 0 or, with paged
    // keys, warp 3" in one expression cost the contiguous E4M3 kernel 2.4%.)
    // ------------------------------------------------------- K-tile producer
    // Lane 0 waits and issues the TMA; for MX formats all lanes also copy the
    // tile's 128 key scale words (word of key m = 32c + lane to row `lane`,
    // word c of the 16-byte rows the TMEM copy reads); for paged keys all
    // lanes hold block-table entries (page_entry), and warps 0 and 3 each
    // issue one of the tile's two 64-key boxes (box `half`), each with its
    // own arrival and byte count on the stage's barrier: one thread issuing
    // 8 KB boxes cannot keep enough of them in flight to stream HBM.
    const int half = PAGED && warp == 3 ? 1 : 0;
    constexpr bool kWarpWide = T::kMX || PAGED;
    // MX: a tile's key scale words come in one bulk copy on the tile's own
    // barrier (put in copy order beforehand), or per key with SF_KEYS.
    constexpr bool sf_bulk = T::kMX && !SF_KEYS;
    const int sf_tiles = (p.N + kKeysPerTile - 1) / kKeysPerTile;
    if (lane == 0) prefetch_tmap(&p.tmap_k);
    // K is re-read by every row-block of its batch: kept in L2 (evict_last),
    // except where a batch has at most two row-blocks (decode), whose keys are
    // read once and would only crowd L2 (measured: contiguous decode 59 -> 55
    // µs, BF16 paged decode 91 -> 84 µs).
    const uint64_t pol_k = p.blocks_per_batch <= 2 ? policy_evict_first() : policy_evict_last();
    // Paged keys: the unit's table entries, 32 per load, lane l holding
    // entry `win` + l (`cur`) and `win` + 32 + l (`nxt`). The next 32 are
    // requested on entering a window, so the table's latency is spread over
    // the tiles of 32 entries instead of stalling every TMA issue.
    const int n_entries = PAGED ? page_index(p, p.N - 1) + 1 : 0;
    const int32_t* table = nullptr;
    int win = 0, cur = 0, nxt = 0;
    auto fetch_entry = [&](int e) { return e < n_entries ? __ldg(table + e) : 0; };
    auto page_entry = [&](int e) {  // warp-collective; e warp-uniform, e >= win
      if (e >= win + 32) {
        if (e < win + 64) {
          cur = nxt;
          win += 32;
        } else {
          win = e;
          cur = fetch_entry(win + lane);
        }
        nxt = fetch_entry(win + 32 + lane);
      }
      return clampi(__shfl_sync(0xffffffffu, cur, e - win), 0, p.num_pages - 1);
    };
    uint32_t kiter = 0;
    for (uint32_t it = 0;; ++it) {
      const int slot = it & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&q_full[slot], (it >> 1) & 1, abort_flag, p.timeout_ns);
      if constexpr (kWarpWide) {
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();  // lane 0's acquire covers the QInfo the other lanes read
      }
      if (!ok) {
        if (lane == 0) raise_error(p.scratch, abort_flag, kErrTimeout);
        break;
      }
      // Read once, at the unit's start: the slot's Q half is refilled only
      // after the MMAs of this unit, which consume every tile loaded here.
      const QInfo& qi = qinfo[slot];
      if (qi.stop) break;
      const int c0 = qi.c0, c1 = qi.c1, b = qi.b;
      if constexpr (PAGED) {
        table = p.block_table + static_cast<int64_t>(b) * p.table_stride;
        win = page_index(p, c0 * kKeysPerTile);
        cur = unit_pages[slot * 32 + lane];  // the scheduler's copy of entry win + lane
        nxt = fetch_entry(win + 32 + lane);
      }
      for (int t = first_tile<MODE>(c0); t < c1; t = next_tile<MODE>(t), ++kiter) {
        const int st = kiter % T::kStages;
        // Rows of this warp's 64-key box (keys 64*half.. of the tile), inside
        // one page (page_size is a multiple of 64). The first box starts
        // below N; a second box wholly past N re-reads the first one's rows
        // (keys no window reads).
        int prow[2] = {0, 0};
        if constexpr (PAGED) {
          const int k0 = t * kKeysPerTile + 64 * half;
          const int kk = k0 < p.N ? k0 : k0 - 64;
          const int e = page_index(p, kk);
          prow[0] = page_entry(e) * p.page_size + (kk - e * p.page_size);
        }
        if (lane == 0)
          ok = mbar_wait(&k_empty[st], ((kiter / T::kStages) & 1) ^ 1, abort_flag, p.timeout_ns);
        if constexpr (kWarpWide) ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&k_full[st], (PAGED ? L::kKTileBytes / 2 : L::kKTileBytes) +
                                                 (sf_bulk && half == 0 ? kSfaBytes : 0));
          if constexpr (sf_bulk)
            if (half == 0)
              bulk_load(sfa_s + st * kSfaBytes,
                        p.k_sf_tiles + (static_cast<int64_t>(b) * sf_tiles + t) * kSfaBytes,
                        kSfaBytes, &k_full[st]);
          uint8_t* kdst = kbuf + st * L::kKTileBytes;
          if constexpr (!PAGED) {
#pragma unroll
            for (int pnl = 0; pnl < L::kPanels; ++pnl)
              tma_load_3d(kdst + pnl * L::kKPanelBytes, &p.tmap_k, &k_full[st],
                          pnl * (T::kSwizzleBytes / T::kTmaElemBytes), t * kKeysPerTile, b, pol_k);
          } else {
#pragma unroll
            for (int pnl = 0; pnl < L::kPanels; ++pnl)
              tma_load_2d(kdst + pnl * L::kKPanelBytes + half * 64 * T::kSwizzleBytes, &p.tmap_k,
                          &k_full[st], pnl * (T::kSwizzleBytes / T::kTmaElemBytes), prow[0],
                          pol_k);
          }
        }
        if constexpr (T::kMX && SF_KEYS) {
          uint8_t* dst = sfa_s + st * kSfaBytes + 16 * lane;
          const uint8_t* src = p.k_sf + (static_cast<int64_t>(b) * p.N + t * kKeysPerTile) * 4;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int m = 32 * c + lane;
            if (t * kKeysPerTile + m < p.N) cp_async_4(dst + 4 * c, src + 4 * m);
          }
          cp_async_arrive(&sf_full[st]);
        }
      }
      if (!ok) {
        if (lane == 0) raise_error(p.scratch, abort_flag, kErrTimeout);
        break;
      }
    }
    if (*abort_flag && lane == 0) {
      // Let the key tiles (and scale copies) of the last kStages issues land
      // before the CTA exits.
      for (uint32_t j = kiter > T::kStages ? kiter - T::kStages : 0; j < kiter; ++j) {
        mbar_wait_drain(&k_full[j % T::kStages], (j / T::kStages) & 1, p.timeout_ns);
        if constexpr (T::kMX && SF_KEYS)
          mbar_wait_drain(&sf_full[j % T::kStages], (j / T::kStages) & 1, p.timeout_ns);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // --------------------------------------------------------------- MMA issuer
    uint32_t kiter = 0, aiter = 0, units_mma = 0;
    // ReLU(s*x) = |s| * max(-x, 0) for s < 0: negate the A operand (bit 13),
    // except where the epilogue applies the sign (NEG_EPI).
    const uint32_t idesc = L::kIdesc | (!NEG_EPI && p.sm_scale < 0.f ? (1u << 13) : 0u);
    // K-major operands, 8-row groups one swizzle atom apart; layout code
    // 2 = 128-byte swizzle, 4 = 64-byte swizzle.
    constexpr uint32_t kLayout = T::kSwizzleBytes == 128 ? 2u : 4u;
    const uint64_t k_desc0 = smem_desc(smem_u32(kbuf), L::kAtomBytes, kLayout);
    const uint64_t q_desc0 = smem_desc(smem_u32(qbuf), L::kAtomBytes, kLayout);
    // Scale factors: 32 rows x 16 bytes, no swizzle, 8-row groups 128 bytes apart.
    const uint64_t sfa_desc0 = smem_desc(smem_u32(sfa_s), 128, 0);
    const uint64_t sfb_desc0 = smem_desc(smem_u32(sfb_s), 128, 0);
    for (uint32_t it = 0;; ++it) {
      const int slot = it & 1;
      if (!mbar_wait(&q_full[slot], (it >> 1) & 1, abort_flag, p.timeout_ns)) {
        raise_error(p.scratch, abort_flag, kErrTimeout);
        break;
      }
      const QInfo& qi = qinfo[slot];
      if (qi.stop) break;
      const int c0 = qi.c0, c1 = qi.c1;
      const int tf = first_tile<MODE>(c0);  // the unit's first tile in this mode
      const uint64_t b_base = q_desc0 + ((slot * L::kQBlockBytes) >> 4);
      bool ok = true;
      for (int t = tf; t < c1; t = next_tile<MODE>(t), ++kiter, ++aiter) {
        const int st = kiter % T::kStages;
        const int acc = aiter % kAccBufs;
        const uint32_t kpar = (kiter / T::kStages) & 1;
        const uint32_t apar = ((aiter / kAccBufs) & 1) ^ 1;
        if (!mbar_wait(&k_full[st], kpar, abort_flag, p.timeout_ns) ||
            (T::kMX && SF_KEYS && !mbar_wait(&sf_full[st], kpar, abort_flag, p.timeout_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sfa = 0, sfb = 0;
        if constexpr (T::kMX) {
          // Scale factors go to TMEM before the accumulator wait, so the copy
          // is off the critical path: slots alternate (key scales by tile, Q
          // scales by unit with tiles), and the slot written here was last
          // read by the MMAs of tile t-2 or earlier, which finished before
          // tile t-1's accumulator could be handed back and its MMAs issued.
          // Copies and MMAs of this thread run in issue order. The scale
          // words were written by cp.async (key scales) and plain stores (Q
          // scales), both generic proxy; the TMEM copy reads them through
          // the async proxy.
          fence_proxy_async_smem();
          sfa = tmem_base + kSfaCol + 4 * (kiter & 1);
          sfb = tmem_base + kSfbCol + 8 * (units_mma & 1);
          if (t == tf) {
            const uint64_t d = sfb_desc0 + ((slot * kSfbBytes) >> 4);
            tc_cp_32x128b_warpx4(sfb, d);
            tc_cp_32x128b_warpx4(sfb + 4, d + (512 >> 4));
          }
          tc_cp_32x128b_warpx4(sfa, sfa_desc0 + ((st * kSfaBytes) >> 4));
        }
        // Sleep until the accumulator is handed back, also with a single
        // accumulator, where the wait is on the critical path: a polling
        // thread takes issue slots from the epilogue warps on its scheduler,
        // whose arithmetic is the longer part of the chain (measured: a
        // polling wait made the MXFP8 kernel 5% slower).
        if (!mbar_wait(&acc_empty[acc], apar, abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // Descriptors differ only in the start-address field (bits 0-13,
        // address >> 4), so every step is the stage/slot base plus an offset.
        const uint64_t a_base = k_desc0 + ((st * L::kKTileBytes) >> 4);
        const uint32_t d_tmem = tmem_base + acc * L::kBlockNR;
#pragma unroll
        for (int kk = 0; kk < L::kSteps; ++kk) {
          const uint32_t pnl = kk / L::kStepsPerPanel, step = kk % L::kStepsPerPanel;
          const uint32_t off = pnl * L::kKPanelBytes + step * kStepBytes;
          const uint32_t offq = pnl * L::kQPanelBytes + step * kStepBytes;
          const uint32_t sf_id = kk * T::kSfIdStep;
          const uint32_t id = T::kMX ? (idesc | (sf_id << 4) | (sf_id << 29)) : idesc;
          mma_step<T::kKind>(d_tmem, a_base + (off >> 4), b_base + (offq >> 4), id,
                             kk > 0 ? 1u : 0u, sfa, sfb);
        }
        tc_commit(&k_empty[st]);
        tc_commit(&acc_full[acc]);
      }
      if (tf < c1) ++units_mma;
      if (!ok) {
        raise_error(p.scratch, abort_flag, kErrTimeout);
        break;
      }
      // The slot's Q half (Q block, Q scales, QInfo) is free once these MMAs
      // and scale copies are done.
      tc_commit(&q_empty[slot]);
    }
    if (*abort_flag) {
      // A commit tracks every MMA and TMEM copy this thread issued: wait for
      // them before the accumulator memory is freed.
      tc_commit(drain);
      mbar_wait_drain(drain, 0, p.timeout_ns);
    }
  } else if (warp >= kEpiWarp0) {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM sub-partition of this warp
    // Groups of warps (one with RB = 4) take alternate tiles: group g the
    // tiles whose index over all units (aiter) is g mod kGroups.
    // (Both are compile-time constants with one group, so the four-row
    // kernels keep no extra live register in their tile loop.)
    constexpr int kWR = R * kSeq;        // rows per warp
    constexpr int kWarpRows = RB / kWR;  // warps per sub-partition in a group
    const int wrow = (warp - kEpiWarp0) >> 2;
    const int grp = kGroups > 1 ? wrow / kWarpRows : 0;
    const int r0 = kWR * (kGroups > 1 ? wrow % kWarpRows : wrow);  // rows r0 .. r0 + kWR - 1
    const int tid128 = quarter * 32 + lane;        // index among the rows' 4 warps
    // The MMA delivers x = s_sign * q.k (negated A for s < 0), so the sum is
    // scaled by |s|; with NEG_EPI the epilogue sums min(x, 0) and scales by s.
    const float sm_abs = NEG_EPI ? p.sm_scale : fabsf(p.sm_scale);
    const float ninf = __int_as_float(0xff800000);
    uint32_t aiter = 0;
    for (uint32_t it = 0;; ++it) {
      const int slot = it & 1;
      if (!mbar_wait(&unit_full[slot], (it >> 1) & 1, abort_flag, p.timeout_ns)) {
        raise_error(p.scratch, abort_flag, kErrTimeout);
        break;
      }
      const UnitInfo& in = info[slot];
      if (in.stop) break;
      const int b = in.b, c0 = in.c0, c1 = in.c1, t0 = in.t0, t1 = in.t1, flags = in.flags;
      int lo[kWR], hi[kWR];
      // Rows past S (a partial last block) are a suffix of the block. Such a
      // row aliases the warp's first row, which is stored after it (rows go
      // in reverse below), so only real values land; a warp with no real
      // row stores nothing (its bound is 0).
      char* orow[kWR];
      bool any_row = false;
      constexpr bool obf = OUT_BF16;
      // bytes per output slot: logits, compact sample logits, or candidates
      constexpr int kSlot = obf ? 2 : 4;
      float thr[kWR];      // kModeFilter: the rows' thresholds
      int32_t rowid[kWR];  // kModeFilter: the rows (-1: absent)
#pragma unroll
      for (int r = 0; r < kWR; ++r) {
        lo[r] = in.lo[r0 + r];
        hi[r] = in.hi[r0 + r];
        const int row = in.row[r0 + r];
        orow[r] = row < 0 ? (r > 0 ? orow[0] : nullptr)
                          : static_cast<char*>(p.out) +
                                static_cast<int64_t>(row) * p.out_row_stride * kSlot;
        any_row |= row >= 0;
        rowid[r] = row;
        if constexpr (MODE == kModeFilter) thr[r] = row >= 0 ? __ldg(p.thr + row) : 0.f;
      }
      const int store_lim = any_row ? p.N : 0;
      const float* wrows = reinterpret_cast<const float*>(wbuf + slot * L::kWBytes) + r0 * kHeads;
      // Compact sample column of the first key of tile t (kModeSample).
      auto sample_col = [](int t) { return first_tile<kModeSample>(t) / kSampleEvery * kKeysPerTile; };
      if (p.clean && (flags & 1) && MODE != kModeFilter && grp == 0) {
        const int end = MODE == kModeSample ? sample_col(t0) : t0 * kKeysPerTile;
#pragma unroll
        for (int r = 0; r < kWR; ++r)
          if (orow[r] != nullptr) fill_neg_inf(orow[r], 0, end, tid128, obf);
      }
      // Per-key scale (E4M3), loaded one tile ahead so that its latency
      // overlaps the previous tile instead of stalling the loop head. Paged
      // keys need two dependent loads (page number, then scale): the page
      // number is loaded two tiles ahead, the scale one tile ahead.
      const bool key_scaled = FMT == kFmtE4M3 && p.k_scales != nullptr;
      const float* kscale_b =
          key_scaled && !PAGED ? p.k_scales + static_cast<int64_t>(b) * p.N : nullptr;
      auto load_kscale = [&](int t) {
        const int jj = t * kKeysPerTile + quarter * 32 + lane;
        if (!(key_scaled && t < c1 && jj < p.N)) return 1.f;
        return __ldg(kscale_b + jj);
      };
      auto load_page = [&](int t) {  // page of this thread's key in tile t, or -1
        const int jj = t * kKeysPerTile + quarter * 32 + lane;
        if (!(key_scaled && t < c1 && jj < p.N)) return -1;
        return clampi(__ldg(p.block_table + static_cast<int64_t>(b) * p.table_stride +
                            page_index(p, jj)),
                      0, p.num_pages - 1);
      };
      auto scale_in_page = [&](int t, int page) {
        if (page < 0) return 1.f;
        const int jj = t * kKeysPerTile + quarter * 32 + lane;
        return __ldg(p.k_scales + static_cast<int64_t>(page) * p.page_size +
                     (jj - page_index(p, jj) * p.page_size));
      };
      // This group's first tile of the unit; its later ones are kGroups
      // apart (kGroups > 1 only computes logits, where tiles are consecutive).
      const int tf = first_tile<MODE>(c0) +
                     (kGroups > 1 ? static_cast<int>((grp + kGroups - aiter % kGroups) % kGroups) : 0);
      // The unit's first pages come from the scheduler's copy of its first
      // 32 table entries: no wait for the table at the unit's start.
      auto first_page = [&](int t) {
        const int jj = t * kKeysPerTile + quarter * 32 + lane;
        if (!(key_scaled && t < c1 && jj < p.N)) return -1;
        const int e = page_index(p, jj) - page_index(p, c0 * kKeysPerTile);
        return e < 32 ? clampi(unit_pages[(2 + slot) * 32 + e], 0, p.num_pages - 1) : load_page(t);
      };
      int page_ahead = PAGED ? first_page(tf + kGroups) : -1;
      float kscale_next = PAGED ? scale_in_page(tf, first_page(tf)) : load_kscale(tf);
      bool ok = true;
      if (PAGED && !any_row) {
        // Every row of this warp is past S (a partial last block; decode with
        // 1-2 new tokens per sequence): only hand each accumulator back.
        // Kept to the paged kernels: in the others its mere presence slowed
        // the E4M3 tile loop, and there the absent rows are just computed
        // and not stored.
        for (int t = c0; t < c1; ++t, ++aiter) {
          if (kGroups > 1 && static_cast<int>(aiter % kGroups) != grp) continue;
          if (!mbar_wait(&acc_full[aiter % kAccBufs], (aiter / kAccBufs) & 1, abort_flag,
                         p.timeout_ns)) {
            ok = false;
            break;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[aiter % kAccBufs]);
        }
      } else {
        for (int t = first_tile<MODE>(c0); t < c1; t = next_tile<MODE>(t), ++aiter) {
          if (kGroups > 1 && static_cast<int>(aiter % kGroups) != grp) continue;
          const int acc = aiter % kAccBufs;
          const int j = t * kKeysPerTile + quarter * 32 + lane;
          const float kscale = kscale_next;
          if constexpr (PAGED) {
            kscale_next = scale_in_page(t + kGroups, page_ahead);
            page_ahead = load_page(t + 2 * kGroups);
          } else {
            kscale_next = load_kscale(kGroups > 1 ? t + kGroups : next_tile<MODE>(t));
          }
          if (!mbar_wait(&acc_full[acc], (aiter / kAccBufs) & 1, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          __syncwarp();  // tcgen05.ld is warp-collective: converge first
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                 acc * L::kBlockNR + r0 * kHeads;
          if constexpr (kSeq > 1) {
            // Row sets last first (an absent row aliases the warp's first
            // row, which must be stored last); the accumulator goes back once
            // the last set is loaded.
#pragma unroll
            for (int sq = kSeq - 1; sq >= 0; --sq) {
              uint32_t v[R][64];
              RowAcc<NEG_EPI, T::kReluAllAdd> racc[R];
#pragma unroll
              for (int r = 0; r < R; ++r) racc[r].zero();
#pragma unroll
              for (int r = 0; r < R; ++r) tmem_ld_64cols(taddr + (sq * R + r) * kHeads, v[r]);
              if (sq == 0) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[acc]);
              }
              head_steps<0, kHeads / 4>(racc, v, wrows + sq * R * kHeads);
              if (j < store_lim) {
#pragma unroll
                for (int r = R - 1; r >= 0; --r) {
                  const int rr = sq * R + r;
                  const float x = racc[r].total();
                  const float v = (j >= lo[rr] && j < hi[rr]) ? x * (sm_abs * kscale) : ninf;
                  if (obf)
                    st_cs_b16(orow[rr] + 2 * static_cast<int64_t>(j), f32_to_bf16_rn(v));
                  else
                    __stcs(reinterpret_cast<float*>(orow[rr]) + j, v);
                }
              }
            }
            continue;
          }
          // Read the rows' 64 columns each, hand the accumulator back, reduce.
          uint32_t v[R][64];
          RowAcc<NEG_EPI, T::kReluAllAdd> racc[R];
#pragma unroll
          for (int r = 0; r < R; ++r) racc[r].zero();
#pragma unroll
          for (int r = 0; r < R; ++r) tmem_ld_64cols(taddr + r * kHeads, v[r]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[acc]);
          head_steps<0, kHeads / 4>(racc, v, wrows);
          float sums[R];
#pragma unroll
          for (int r = 0; r < R; ++r) sums[r] = racc[r].total();
          if constexpr (MODE == kModeLogits) {
            if (j < store_lim) {
#pragma unroll
              for (int r = R - 1; r >= 0; --r) {
                const float v = (j >= lo[r] && j < hi[r]) ? sums[r] * (sm_abs * kscale) : ninf;
                if (obf)
                  st_cs_b16(orow[r] + 2 * static_cast<int64_t>(j), f32_to_bf16_rn(v));
                else
                  __stcs(reinterpret_cast<float*>(orow[r]) + j, v);
              }
            }
          } else if constexpr (MODE == kModeSample) {
            // every compact column of a sample tile is written: -inf past N
            if (any_row) {
              const int col = t / kSampleEvery * kKeysPerTile + quarter * 32 + lane;
#pragma unroll
              for (int r = R - 1; r >= 0; --r) {
                const float v = (j < p.N && j >= lo[r] && j < hi[r]) ? sums[r] * (sm_abs * kscale)
                                                                     : ninf;
                __stcs(reinterpret_cast<float*>(orow[r]) + col, v);
              }
            }
          } else {
            // Keep the in-window values >= the row's threshold, packed at the
            // front of the group's 32 slots in key order (the value of the
            // key of mask bit l is at the rank of bit l among the set bits),
            // and the group's mask word; no atomics: slots and word belong
            // to this (row, tile, quarter) alone. Packing lets the merge read
            // one sector per group instead of most of the group's line.
            const int grp = (t - t / kSampleEvery - 1) * 4 + quarter;
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const float v = sums[r] * (sm_abs * kscale);
              const bool pass = rowid[r] >= 0 && j < p.N && j >= lo[r] && j < hi[r] && v >= thr[r];
              const uint32_t m = __ballot_sync(0xffffffffu, pass);
              if (pass)
                reinterpret_cast<float*>(orow[r])[grp * 32 + __popc(m & ((1u << lane) - 1u))] = v;
              if (lane == 0 && m != 0u)
                p.mask[static_cast<int64_t>(rowid[r]) * p.mask_row_stride + grp] = m;
            }
          }
        }
      }
      if (!ok) {
        raise_error(p.scratch, abort_flag, kErrTimeout);
        break;
      }
      if (p.clean && (flags & 2) && MODE != kModeFilter && grp == 0) {
        const int from = MODE == kModeSample ? sample_col(t1) : t1 * kKeysPerTile;
        const int to = MODE == kModeSample ? static_cast<int>(p.out_row_stride) : p.N;
#pragma unroll
        for (int r = 0; r < kWR; ++r)
          if (orow[r] != nullptr) fill_neg_inf(orow[r], from, to, tid128, obf);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&unit_empty[slot]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0) {
    // Last CTA out resets the unit counter for the next call on this stream.
    __threadfence();
    const int prev = atomicAdd(p.scratch + 1, 1);
    if (prev == static_cast<int>(gridDim.x) - 1) {
      atomicExch(p.scratch + 0, 0);
      atomicExch(p.scratch + 1, 0);
      __threadfence();
    }
  }
}

// Diagnostic: one wait of the kind every role above uses, on a barrier that
// nothing arrives on, so that it runs out after `timeout_ns`; it records
// kErrTimeout in the error word exactly as a role that gives up does. Nothing
// is in flight when the kernel returns, so the context stays usable.
__global__ void wait_selftest_kernel(int32_t* scratch, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_word;
  if (threadIdx.x == 0) {
    abort_word = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, &abort_word, timeout_ns)) atomicExch(scratch + 2, kErrTimeout);
  }
}

}  // namespace dsa
