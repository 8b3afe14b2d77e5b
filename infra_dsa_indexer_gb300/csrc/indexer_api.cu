// Host side of the C ABI declared in include/dsa_indexer.h: argument checks,
// TMA tensor maps, per-(device, stream) scratch, the persistent launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "dsa_indexer.h"
#include "indexer_kernel.cuh"
#include "plan_kernel.cuh"
#include "scale_order_kernel.cuh"
#include "topk_kernel.cuh"
#include "window_kernel.cuh"

namespace {

using dsa::KernelParams;

constexpr int kScratchInts = 64;  // 256 bytes per (device, stream)

struct DeviceInfo {
  bool valid = false;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  // per kernel instantiation: format, mode, sign, output type, paging (and,
  // from 128 on, the two-row-block BF16/E4M3 kernels, from 136 on the MX
  // kernels that copy key scales per key)
  bool smem_set[144] = {};
  bool plan_attr_set = false;
};

std::mutex g_mutex;
std::map<int, DeviceInfo> g_devices;
// Scratch of indexer_logits per (device, stream): kScratchInts header words
// ([0] unit counter, [1] finished CTAs, [2] error word), then the row order
// of a grouped call (B*S words).
struct Scratch {
  int32_t* ptr = nullptr;
  int64_t words = 0;
};
std::map<std::pair<int, uintptr_t>, Scratch> g_scratch;
int64_t g_wait_limit_ns = 2000000000LL;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_device_info(int dev, DeviceInfo** out) {
  DeviceInfo& di = g_devices[dev];
  if (!di.valid) {
    if (cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
            cudaSuccess)
      return IDX_ERR_CUDA;
    di.valid = true;
  }
  *out = &di;
  return IDX_OK;
}

int get_encoder() {
  if (g_encode) return IDX_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return IDX_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return IDX_OK;
}

// At least `words` words of scratch for (dev, stream), stream-ordered: the
// block comes from the device's stream-ordered pool (cudaMallocAsync), so
// neither the first allocation nor a later growth waits for the device.
// Growing allocates the larger block on `stream`, carries the error word over
// with a device-to-device copy on `stream` and frees the old block on
// `stream` (after every earlier call on it has finished with it).
int get_scratch(int dev, cudaStream_t stream, int64_t words, int32_t** out) {
  words = std::max<int64_t>(words, kScratchInts);
  Scratch& sc = g_scratch[std::make_pair(dev, reinterpret_cast<uintptr_t>(stream))];
  if (sc.ptr != nullptr && sc.words >= words) {
    *out = sc.ptr;
    return IDX_OK;
  }
  void* raw = nullptr;
  if (cudaMallocAsync(&raw, words * sizeof(int32_t), stream) != cudaSuccess) return IDX_ERR_CUDA;
  int32_t* p = static_cast<int32_t*>(raw);
  if (cudaMemsetAsync(p, 0, kScratchInts * sizeof(int32_t), stream) != cudaSuccess ||
      (sc.ptr != nullptr &&
       (cudaMemcpyAsync(p + 2, sc.ptr + 2, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream) !=
            cudaSuccess ||
        cudaFreeAsync(sc.ptr, stream) != cudaSuccess))) {
    cudaFreeAsync(p, stream);
    return IDX_ERR_CUDA;
  }
  sc.ptr = p;
  sc.words = words;
  *out = p;
  return IDX_OK;
}

// Rows are regrouped by window (one planning launch before the logits
// kernel) when the caller asks for it and the call may allocate.
bool groups_rows(const idx_shape& sh, bool fixed_scratch) {
  return (sh.flags & IDX_FLAG_GROUP_ROWS) != 0 && !fixed_scratch;
}

int launch_plan(const int32_t* ks, const int32_t* ke, const idx_shape& sh, int32_t* perm,
                DeviceInfo* di, cudaStream_t stream) {
  if (!di->plan_attr_set) {
    if (cudaFuncSetAttribute(dsa::plan_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dsa::kPlanSmemBytes) != cudaSuccess)
      return IDX_ERR_CUDA;
    di->plan_attr_set = true;
  }
  dsa::plan_rows_kernel<<<sh.B, dsa::kPlanThreads, dsa::kPlanSmemBytes, stream>>>(ks, ke, sh.S,
                                                                                  sh.N, perm);
  return cudaGetLastError() == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

// Words of scratch one call uses: [0] unit counter, [1] finished CTAs,
// [2] device error word.
constexpr int kScratchWordsPerCall = 3;

// Scratch of indexer_logits_noalloc: a fixed array in the library's device
// image (every GPU that loads the library holds these 256 bytes until the
// process exits). Host code may not use its name as a pointer: its device
// address is looked up once per device with cudaGetSymbolAddress.
constexpr int kFixedScratchWords = 64;
constexpr int kMaxDevices = 64;
__device__ __align__(256) int32_t g_fixed_scratch[kFixedScratchWords];
int32_t* g_fixed_scratch_addr[kMaxDevices] = {};

// Called with g_mutex held and `dev` current.
int get_fixed_scratch(int dev, int32_t** out) {
  if (dev < 0 || dev >= kMaxDevices) return IDX_ERR_DEVICE;
  if (g_fixed_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_fixed_scratch) != cudaSuccess || ptr == nullptr)
      return IDX_ERR_CUDA;
    g_fixed_scratch_addr[dev] = static_cast<int32_t*>(ptr);
  }
  *out = g_fixed_scratch_addr[dev];
  return IDX_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D or 3-D tiled map. dims/strides in elements/bytes.
int encode_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int rank,
               const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
               CUtensorMapSwizzle swizzle) {
  uint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, dtype, rank, const_cast<void*>(base), dims, strides_bytes, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IDX_OK : IDX_ERR_CUDA;
}

// Launches a selection kernel (it starts with griddepcontrol.wait) as a
// programmatic dependent of the previous kernel on the stream: its blocks may
// be placed while that kernel finishes, and read its output only after it
// has completed.
template <typename... KArgs, typename... Args>
int launch_dependent(void (*kernel)(KArgs...), unsigned grid, unsigned block, cudaStream_t stream,
                     Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

template <int FMT, bool NEG_EPI, bool OUT_BF16, bool PAGED, int MODE = dsa::kModeLogits,
          int RB = dsa::kRowsPerBlock, bool SF_KEYS = false>
int launch_kernel(const KernelParams& prm, int grid, DeviceInfo* di, cudaStream_t stream) {
  constexpr int smem = dsa::Layout<FMT, RB>::kBytes;
  auto kern = dsa::indexer_logits_kernel<FMT, NEG_EPI, OUT_BF16, PAGED, MODE, RB, SF_KEYS>;
  static_assert(RB == dsa::kRowsPerBlock || FMT < 2, "two-row blocks: BF16 and E4M3");
  bool& attr_set =
      di->smem_set[SF_KEYS ? 136 + (FMT - 2) * 4 + (NEG_EPI ? 2 : 0) + (OUT_BF16 ? 1 : 0)
                   : RB == dsa::kRowsPerBlock
                       ? FMT * 32 + MODE * 8 + (NEG_EPI ? 4 : 0) + (OUT_BF16 ? 2 : 0) +
                             (PAGED ? 1 : 0)
                       : 128 + FMT * 4 + (OUT_BF16 ? 2 : 0) + (PAGED ? 1 : 0)];
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return IDX_ERR_CUDA;
    attr_set = true;
  }
  kern<<<grid, dsa::Layout<FMT, RB>::kThreads, smem, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

// Query rows per block of a call: 2 for BF16/E4M3 logits whose batches have
// at most two rows (decode), where four-row blocks would leave half of each
// MMA and of the epilogue warps without a row; else kRowsPerBlock.
int rows_per_block(const idx_shape& sh, int mode, bool grouped) {
  const bool two = (sh.fmt == IDX_FMT_BF16 || sh.fmt == IDX_FMT_E4M3) && sh.S <= 2 &&
                   mode == dsa::kModeLogits && !grouped;
  return two ? 2 : dsa::kRowsPerBlock;
}

template <int FMT, bool NEG_EPI>
int launch(const KernelParams& prm, int grid, DeviceInfo* di, cudaStream_t stream, int mode,
           int rb) {
  if constexpr (FMT == dsa::kFmtBF16 || FMT == dsa::kFmtE4M3) {
    if (rb == 2) {
      constexpr int kM = dsa::kModeLogits;
      if (prm.block_table != nullptr)
        return prm.out_bf16 ? launch_kernel<FMT, false, true, true, kM, 2>(prm, grid, di, stream)
                            : launch_kernel<FMT, false, false, true, kM, 2>(prm, grid, di, stream);
      return prm.out_bf16 ? launch_kernel<FMT, false, true, false, kM, 2>(prm, grid, di, stream)
                          : launch_kernel<FMT, false, false, false, kM, 2>(prm, grid, di, stream);
    }
  }
  if constexpr (FMT == dsa::kFmtMXFP8 || FMT == dsa::kFmtMXFP4) {
    // No key scales in copy order (no library scratch): per-key copies.
    if (prm.k_sf_tiles == nullptr) {
      if (mode != dsa::kModeLogits || prm.block_table != nullptr) return IDX_ERR_UNSUPPORTED;
      constexpr int kM = dsa::kModeLogits, kR = dsa::kRowsPerBlock;
      return prm.out_bf16
                 ? launch_kernel<FMT, NEG_EPI, true, false, kM, kR, true>(prm, grid, di, stream)
                 : launch_kernel<FMT, NEG_EPI, false, false, kM, kR, true>(prm, grid, di, stream);
    }
  }
  if (mode == dsa::kModeSample)
    return launch_kernel<FMT, NEG_EPI, false, false, dsa::kModeSample>(prm, grid, di, stream);
  if (mode == dsa::kModeFilter)
    return launch_kernel<FMT, NEG_EPI, false, false, dsa::kModeFilter>(prm, grid, di, stream);
  if (prm.block_table != nullptr)
    return prm.out_bf16 ? launch_kernel<FMT, NEG_EPI, true, true>(prm, grid, di, stream)
                        : launch_kernel<FMT, NEG_EPI, false, true>(prm, grid, di, stream);
  return prm.out_bf16 ? launch_kernel<FMT, NEG_EPI, true, false>(prm, grid, di, stream)
                      : launch_kernel<FMT, NEG_EPI, false, false>(prm, grid, di, stream);
}

}  // namespace

extern "C" {

int indexer_version(void) { return 200; }

int indexer_launches_per_call(const idx_shape* shape) {
  if (shape == nullptr) return 1;
  const bool mx = shape->fmt == IDX_FMT_MXFP8 || shape->fmt == IDX_FMT_MXFP4;
  return 1 + (groups_rows(*shape, false) ? 1 : 0) + (mx ? 1 : 0);
}

const char* indexer_status_string(int status) {
  switch (status) {
    case IDX_OK: return "ok";
    case IDX_ERR_NULL: return "a required pointer is NULL";
    case IDX_ERR_SHAPE: return "unsupported or inconsistent shape (H must be 64, D 128, B, S, N >= 1, out_row_stride >= N)";
    case IDX_ERR_FORMAT: return "unknown format, or scales missing/present for the wrong format";
    case IDX_ERR_ALIGN:
      return "q/k/w base address or q/k stride is not 16-byte aligned, or out is not aligned "
             "to its element size";
    case IDX_ERR_SCALE: return "sm_scale is not finite";
    case IDX_ERR_DEVICE: return "current device is not compute capability 10.3 (sm_103)";
    case IDX_ERR_CUDA: return "a CUDA runtime call failed";
    case IDX_ERR_TIMEOUT: return "a device-side wait ran out; the output of that call is invalid";
    case IDX_ERR_UNSUPPORTED: return "request not supported by this build";
    case IDX_ERR_SCRATCH:
      return "call needs more scratch than the fixed no-allocation array (or the workspace "
             "given) holds";
    default: return "unknown status";
  }
}

int64_t indexer_set_wait_limit_ns(int64_t ns) {
  std::lock_guard<std::mutex> lock(g_mutex);
  const int64_t prev = g_wait_limit_ns;
  g_wait_limit_ns = ns < 1000000 ? 1000000 : ns;
  return prev;
}

}  // extern "C"

namespace {

// One pass of the fused top-k call (see indexer_logits_topk): which mode,
// its per-row thresholds and candidate counts, and whether the row order of
// a grouped call is already planned (by the pass before).
struct PassArgs {
  int mode = dsa::kModeLogits;
  const float* thr = nullptr;
  uint32_t* mask = nullptr;
  int64_t mask_row_stride = 0;
  int64_t out_row_stride = 0;  // overrides the shape's (elements or candidate slots)
  bool planned = false;
};

// Validate, build the tensor maps and launch one call. `fixed_scratch` is
// false for indexer_logits (scratch per (device, stream), allocated on first
// use) or selects the no-allocation variant's fixed device array. `paged` is
// null for contiguous keys.
int enqueue_logits(const void* q, const uint8_t* q_sf, const void* k, const uint8_t* k_sf,
                   const float* k_scales, const void* w, const int32_t* ks, const int32_t* ke,
                   float sm_scale, int clean, void* out, const idx_shape* shape,
                   cudaStream_t stream, bool fixed_scratch, const idx_paged* paged = nullptr,
                   const PassArgs& pass = PassArgs()) {
  if (!shape || !q || !k || !w || !ks || !ke || !out) return IDX_ERR_NULL;
  const idx_shape sh = *shape;
  idx_paged pg{};
  if (paged) {
    pg = *paged;
    if (!pg.block_table) return IDX_ERR_NULL;
    if (pg.page_size < 64 || pg.page_size % 64 != 0 || pg.num_pages < 1 || pg.reserved != 0 ||
        sh.k_batch_bytes != 0 || sh.N < 1 ||
        pg.table_stride < (static_cast<int64_t>(sh.N) + pg.page_size - 1) / pg.page_size ||
        static_cast<int64_t>(pg.num_pages) * pg.page_size >= (int64_t(1) << 31))
      return IDX_ERR_SHAPE;
  }
  if (sh.fmt < IDX_FMT_BF16 || sh.fmt > IDX_FMT_MXFP4) return IDX_ERR_FORMAT;
  if (sh.w_fmt != IDX_W_F32 && sh.w_fmt != IDX_W_BF16) return IDX_ERR_FORMAT;
  const bool mx = sh.fmt == IDX_FMT_MXFP8 || sh.fmt == IDX_FMT_MXFP4;
  if (mx && (!q_sf || !k_sf)) return IDX_ERR_NULL;
  if (!mx && (q_sf || k_sf)) return IDX_ERR_FORMAT;
  if (k_scales && sh.fmt != IDX_FMT_E4M3) return IDX_ERR_FORMAT;
  if (sh.H != dsa::kHeads || sh.D != dsa::kHeadDim || (sh.flags & ~(IDX_FLAG_GROUP_ROWS | IDX_FLAG_OUT_BF16)) != 0)
    return IDX_ERR_SHAPE;
  if (sh.B < 1 || sh.S < 1 || sh.N < 1) return IDX_ERR_SHAPE;
  if (!std::isfinite(sm_scale)) return IDX_ERR_SCALE;

  const int64_t elem_row_bytes =
      sh.fmt == IDX_FMT_BF16 ? 2 * sh.D : (sh.fmt == IDX_FMT_MXFP4 ? sh.D / 2 : sh.D);
  const int64_t q_row = sh.q_row_bytes ? sh.q_row_bytes : elem_row_bytes;
  const int64_t k_row = sh.k_row_bytes ? sh.k_row_bytes : elem_row_bytes;
  const int64_t k_batch = sh.k_batch_bytes ? sh.k_batch_bytes : k_row * sh.N;
  const int64_t out_stride =
      pass.mode != dsa::kModeLogits ? pass.out_row_stride
                                    : (sh.out_row_stride ? sh.out_row_stride : sh.N);
  if (q_row < elem_row_bytes || k_row < elem_row_bytes || k_batch < k_row * sh.N ||
      (pass.mode == dsa::kModeLogits && out_stride < sh.N))
    return IDX_ERR_SHAPE;
  const int64_t total_rows = static_cast<int64_t>(sh.B) * sh.S;
  if (total_rows * sh.H >= (int64_t(1) << 31) || static_cast<int64_t>(sh.B) * sh.N >= (int64_t(1) << 31))
    return IDX_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(w) || q_row % 16 || k_row % 16 ||
      k_batch % 16)
    return IDX_ERR_ALIGN;
  if (mx && ((reinterpret_cast<uintptr_t>(q_sf) & 3u) || (reinterpret_cast<uintptr_t>(k_sf) & 3u)))
    return IDX_ERR_ALIGN;
  const bool out_bf16 = (sh.flags & IDX_FLAG_OUT_BF16) != 0;
  if (reinterpret_cast<uintptr_t>(out) & (out_bf16 ? 1u : 3u)) return IDX_ERR_ALIGN;

  std::lock_guard<std::mutex> lock(g_mutex);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ERR_CUDA;
  DeviceInfo* di = nullptr;
  int st = get_device_info(dev, &di);
  if (st) return st;
  if (di->cc_major != 10 || di->cc_minor != 3) return IDX_ERR_DEVICE;
  if ((st = get_encoder())) return st;
  int32_t* scratch = nullptr;
  // MX key scale words in copy order (scale_order_kernel), 128 words per
  // (batch, key tile), after the header words and the row order; not with
  // the fixed array (the kernel then copies them per key).
  const bool sf_order = (sh.fmt == IDX_FMT_MXFP8 || sh.fmt == IDX_FMT_MXFP4) && !fixed_scratch;
  const int64_t key_tiles = (static_cast<int64_t>(sh.N) + dsa::kKeysPerTile - 1) / dsa::kKeysPerTile;
  const int64_t sf_off =
      (kScratchInts + (groups_rows(sh, fixed_scratch) ? total_rows : 0) + 63) / 64 * 64;
  const int64_t sf_words = sf_order ? static_cast<int64_t>(sh.B) * key_tiles * 128 : 0;
  if (fixed_scratch) {
    if ((st = get_fixed_scratch(dev, &scratch))) return st;
    // The array keeps the previous call's words: start this one from zero.
    if (cudaMemsetAsync(scratch, 0, kScratchWordsPerCall * sizeof(int32_t), stream) != cudaSuccess)
      return IDX_ERR_CUDA;
  } else if ((st = get_scratch(dev, stream, sf_order ? sf_off + sf_words : sf_off, &scratch))) {
    return st;
  }

  KernelParams prm;
  std::memset(&prm, 0, sizeof(prm));
  const CUtensorMapDataType dt =
      sh.fmt == IDX_FMT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  // One box spans one swizzle panel: 128 bytes (64-byte for packed E2M1 rows).
  const bool fp4 = sh.fmt == IDX_FMT_MXFP4;
  const uint32_t panel_elems = sh.fmt == IDX_FMT_BF16 ? 64 : (fp4 ? 64 : 128);
  const CUtensorMapSwizzle swz = fp4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  const uint64_t row_elems = fp4 ? static_cast<uint64_t>(sh.D / 2) : static_cast<uint64_t>(sh.D);
  {
    const uint64_t dims[2] = {row_elems, static_cast<uint64_t>(total_rows * sh.H)};
    const uint64_t strides[1] = {static_cast<uint64_t>(q_row)};
    const uint32_t box[2] = {panel_elems, static_cast<uint32_t>(dsa::kHeads)};  // one row
    if ((st = encode_map(&prm.tmap_q, q, dt, 2, dims, strides, box, swz))) return st;
  }
  {
    if (!paged) {
      const uint64_t dims[3] = {row_elems, static_cast<uint64_t>(sh.N),
                                static_cast<uint64_t>(sh.B)};
      const uint64_t strides[2] = {static_cast<uint64_t>(k_row), static_cast<uint64_t>(k_batch)};
      const uint32_t box[3] = {panel_elems, static_cast<uint32_t>(dsa::kKeysPerTile), 1};
      if ((st = encode_map(&prm.tmap_k, k, dt, 3, dims, strides, box, swz))) return st;
    } else {
      // the whole cache as rows of keys; a box is 64 keys inside one page
      const uint64_t dims[2] = {row_elems,
                                static_cast<uint64_t>(pg.num_pages) * pg.page_size};
      const uint64_t strides[1] = {static_cast<uint64_t>(k_row)};
      const uint32_t box[2] = {panel_elems, 64};
      if ((st = encode_map(&prm.tmap_k, k, dt, 2, dims, strides, box, swz))) return st;
      prm.block_table = pg.block_table;
      prm.page_size = pg.page_size;
      const dsa::PageDiv pdiv = dsa::page_div_make(static_cast<uint32_t>(pg.page_size));
      prm.page_magic = pdiv.magic;
      prm.page_shift = pdiv.shift;
      prm.table_stride = pg.table_stride;
      prm.num_pages = pg.num_pages;
    }
  }
  prm.q_sf = q_sf;
  prm.k_sf = k_sf;
  prm.k_scales = k_scales;
  prm.w = w;
  prm.ks = ks;
  prm.ke = ke;
  prm.out = out;
  prm.out_bf16 = out_bf16 ? 1 : 0;
  prm.thr = pass.thr;
  prm.mask = pass.mask;
  prm.mask_row_stride = pass.mask_row_stride;
  prm.scratch = scratch;
  prm.out_row_stride = out_stride;
  prm.B = sh.B;
  prm.S = sh.S;
  prm.N = sh.N;
  prm.w_bf16 = sh.w_fmt == IDX_W_BF16;
  prm.clean = clean != 0 || pass.mode == dsa::kModeSample;
  prm.sm_scale = sm_scale;
  const int rb = rows_per_block(sh, pass.mode, groups_rows(sh, fixed_scratch));
  prm.blocks_per_batch = (sh.S + rb - 1) / rb;
  prm.timeout_ns = static_cast<uint64_t>(g_wait_limit_ns);

  // Units: every row-block split into nchunk pieces of its key tiles. The
  // base count gives long rows pieces of at most ~64 tiles and small problems
  // enough pieces for about eight per SM; the search below then adjusts it.
  const int64_t row_blocks = static_cast<int64_t>(sh.B) * prm.blocks_per_batch;
  const int64_t tiles_max = (sh.N + dsa::kKeysPerTile - 1) / dsa::kKeysPerTile;
  int64_t nchunk = (tiles_max + 63) / 64;
  const int64_t want = (8 * di->sm_count + row_blocks - 1) / row_blocks;
  nchunk = std::max<int64_t>(nchunk, std::min<int64_t>(want, tiles_max));
  nchunk = std::max<int64_t>(nchunk, 1);
  // Then, among nchunk/2 .. 2*nchunk pieces (at most tiles_max), the count
  // with the shortest estimated run of the persistent grid: rounds of units
  // (ceil(units / SMs)) times the tiles of a unit plus about two tiles' worth
  // of per-unit cost (claim, Q block, windows); ties go to fewer units. A
  // row-block is taken as tiles_max tiles (the host does not read windows),
  // so fewer pieces than nchunk are taken only while the grid still runs at
  // least 16 rounds (unit sizes vary; a short grid's tail does not follow
  // the estimate), or when they fit the whole grid in one round (the
  // 128 x 1024 causal call: 128 two-tile units, 14.5 -> 12.5 µs, against 256
  // one-tile units in two rounds). Measured: 2048 x 32768 calls (2048 units in 13.5 rounds
  // at 4 pieces) take 5 pieces and run 2% faster; 8192 x 65536 calls take 4
  // instead of 8 (-0.4%).
  {
    int64_t best = nchunk, best_cost = INT64_MAX;
    for (int64_t n = (nchunk + 1) / 2; n <= std::min<int64_t>(2 * nchunk, tiles_max); ++n) {
      const int64_t rounds = (row_blocks * n + di->sm_count - 1) / di->sm_count;
      if (n < nchunk && rounds < 16 && rounds > 1) continue;
      const int64_t cost = rounds * ((tiles_max + n - 1) / n + 2);
      if (cost < best_cost) {
        best = n;
        best_cost = cost;
      }
    }
    nchunk = best;
  }
  const int64_t units = row_blocks * nchunk;
  if (units >= (int64_t(1) << 30)) return IDX_ERR_SHAPE;
  prm.nchunk = static_cast<int32_t>(nchunk);
  prm.num_units = static_cast<int32_t>(units);
  const int grid = static_cast<int>(std::min<int64_t>(di->sm_count, units));
  if (groups_rows(sh, fixed_scratch)) {
    prm.perm = scratch + kScratchInts;
    if (!pass.planned &&
        (st = launch_plan(ks, ke, sh, const_cast<int32_t*>(prm.perm), di, stream)))
      return st;
  }
  if (sf_order) {
    uint32_t* sf = reinterpret_cast<uint32_t*>(scratch + sf_off);
    prm.k_sf_tiles = reinterpret_cast<const uint8_t*>(sf);
    // The fused call's second pass reuses the first pass's words.
    if (!pass.planned) {
      const int threads = 256;
      const int64_t blocks = std::min<int64_t>((sf_words + threads - 1) / threads,
                                               static_cast<int64_t>(di->sm_count) * 8);
      dsa::scale_order_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(
          reinterpret_cast<const uint32_t*>(k_sf), sh.N, static_cast<int>(key_tiles), sf_words,
          paged ? pg.block_table : nullptr, paged ? pg.table_stride : 0,
          paged ? pg.page_size : 0, paged ? pg.num_pages : 0, sf);
      if (cudaGetLastError() != cudaSuccess) return IDX_ERR_CUDA;
    }
  }

  const int mode = pass.mode;
  switch (sh.fmt) {
    case IDX_FMT_BF16: return launch<dsa::kFmtBF16, false>(prm, grid, di, stream, mode, rb);
    case IDX_FMT_E4M3: return launch<dsa::kFmtE4M3, false>(prm, grid, di, stream, mode, rb);
    case IDX_FMT_MXFP8: return launch<dsa::kFmtMXFP8, false>(prm, grid, di, stream, mode, rb);
    case IDX_FMT_MXFP4:
      return sm_scale < 0.f ? launch<dsa::kFmtMXFP4, true>(prm, grid, di, stream, mode, rb)
                            : launch<dsa::kFmtMXFP4, false>(prm, grid, di, stream, mode, rb);
    default: return IDX_ERR_UNSUPPORTED;
  }
}

}  // namespace

extern "C" {

int indexer_logits(const void* q, const uint8_t* q_sf, const void* k, const uint8_t* k_sf,
                   const float* k_scales, const void* w, const int32_t* ks, const int32_t* ke,
                   float sm_scale, int clean, void* out, const idx_shape* shape,
                   idx_stream_t stream) {
  return enqueue_logits(q, q_sf, k, k_sf, k_scales, w, ks, ke, sm_scale, clean, out, shape,
                        reinterpret_cast<cudaStream_t>(stream), false);
}

int indexer_logits_noalloc(const void* q, const uint8_t* q_sf, const void* k,
                           const uint8_t* k_sf, const float* k_scales, const void* w,
                           const int32_t* ks, const int32_t* ke, float sm_scale, int clean,
                           void* out, const idx_shape* shape, idx_stream_t stream) {
  // One call needs kScratchWordsPerCall words whatever the shape; refuse
  // anything that would need more than the fixed array holds.
  if (kScratchWordsPerCall > kFixedScratchWords) return IDX_ERR_SCRATCH;
  return enqueue_logits(q, q_sf, k, k_sf, k_scales, w, ks, ke, sm_scale, clean, out, shape,
                        reinterpret_cast<cudaStream_t>(stream), true);
}

int indexer_paged_logits(const void* q, const uint8_t* q_sf, const void* k_cache,
                         const uint8_t* k_sf_cache, const float* k_scales_cache, const void* w,
                         const int32_t* ks, const int32_t* ke, float sm_scale, int clean,
                         void* out, const idx_shape* shape, const idx_paged* paged,
                         idx_stream_t stream) {
  if (!paged) return IDX_ERR_NULL;
  return enqueue_logits(q, q_sf, k_cache, k_sf_cache, k_scales_cache, w, ks, ke, sm_scale, clean,
                        out, shape, reinterpret_cast<cudaStream_t>(stream), false, paged);
}

int indexer_get_last_error(idx_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ERR_CUDA;
  int32_t* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    auto it = g_scratch.find(std::make_pair(dev, reinterpret_cast<uintptr_t>(stream)));
    if (it == g_scratch.end() || it->second.ptr == nullptr) return IDX_OK;
    scratch = it->second.ptr;
  }
  if (cudaStreamSynchronize(stream) != cudaSuccess) return IDX_ERR_CUDA;
  int32_t word = 0;
  if (cudaMemcpy(&word, scratch + 2, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return IDX_ERR_CUDA;
  if (word != 0) {
    const int32_t zero[3] = {0, 0, 0};
    // A run that gave up may leave the unit counter and the CTA count behind.
    if (cudaMemcpy(scratch, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return IDX_ERR_CUDA;
  }
  return word == 0 ? IDX_OK : (word == dsa::kErrTimeout ? IDX_ERR_TIMEOUT : word);
}

int indexer_noalloc_get_last_error(idx_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ERR_CUDA;
  int32_t* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (dev < 0 || dev >= kMaxDevices || g_fixed_scratch_addr[dev] == nullptr) return IDX_OK;
    scratch = g_fixed_scratch_addr[dev];
  }
  if (cudaStreamSynchronize(stream) != cudaSuccess) return IDX_ERR_CUDA;
  int32_t word = 0;
  if (cudaMemcpy(&word, scratch + 2, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return IDX_ERR_CUDA;
  if (word != 0) {
    const int32_t zero[kScratchWordsPerCall] = {0, 0, 0};
    if (cudaMemcpy(scratch, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return IDX_ERR_CUDA;
  }
  return word == 0 ? IDX_OK : (word == dsa::kErrTimeout ? IDX_ERR_TIMEOUT : word);
}

int indexer_stream_release(idx_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  auto it = g_scratch.find(std::make_pair(dev, reinterpret_cast<uintptr_t>(stream)));
  if (it == g_scratch.end()) return IDX_OK;
  const int rc = it->second.ptr == nullptr || cudaFreeAsync(it->second.ptr, stream) == cudaSuccess
                     ? IDX_OK
                     : IDX_ERR_CUDA;
  g_scratch.erase(it);
  return rc;
}

int indexer_topk(const void* logits, int logits_bf16, int64_t rows, int32_t N,
                 int64_t row_stride, int32_t k, int32_t* idx, int64_t idx_stride,
                 idx_stream_t stream_) {
  if (!logits || !idx) return IDX_ERR_NULL;
  if (rows < 1 || rows > 0x7fffffffLL || N < 1 || k < 1 || row_stride < N || idx_stride < k)
    return IDX_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(logits) & (logits_bf16 ? 1u : 3u)) ||
      (reinterpret_cast<uintptr_t>(idx) & 3u))
    return IDX_ERR_ALIGN;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ERR_CUDA;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo* di = nullptr;
    int st = get_device_info(dev, &di);
    if (st) return st;
    if (di->cc_major != 10 || di->cc_minor != 3) return IDX_ERR_DEVICE;
    sms = di->sm_count;
  }
  // One CTA per row; rows that cannot fill the GPU at 512 threads and four
  // CTAs per SM get 1024 threads each. Launched as a programmatic dependent
  // of the previous kernel on the stream (the kernel waits for it first), so
  // its launch overlaps that kernel's end instead of following it.
  const bool few = rows <= 2LL * sms;
  constexpr int kMany = dsa::kTopkThreads, kFew = dsa::kTopkThreadsFew;
  const unsigned grid = static_cast<unsigned>(rows);
  if (logits_bf16)
    return few ? launch_dependent(dsa::topk_rows_kernel<kFew, true>, grid, kFew, stream, logits,
                                  row_stride, N, k, idx, idx_stride)
               : launch_dependent(dsa::topk_rows_kernel<kMany, true>, grid, kMany, stream, logits,
                                  row_stride, N, k, idx, idx_stride);
  return few ? launch_dependent(dsa::topk_rows_kernel<kFew, false>, grid, kFew, stream, logits,
                                row_stride, N, k, idx, idx_stride)
             : launch_dependent(dsa::topk_rows_kernel<kMany, false>, grid, kMany, stream, logits,
                                row_stride, N, k, idx, idx_stride);
}

}  // extern "C"

namespace {

// Layout of the fused top-k call's workspace, each part 256-byte aligned:
// per-row mask words (one per 32 keys of the filtered tiles) and thresholds,
// the compact sample rows, and a value slot for every key of the filtered
// tiles (so no row can overflow it; only kept values are written).
struct TopkWorkspace {
  int64_t rows = 0, ns_cols = 0, cap = 0, mask_stride = 0;
  int64_t off_mask = 0, off_thr = 0, off_s = 0, off_c = 0, bytes = 0;
};

int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

bool topk_workspace(const idx_shape& sh, TopkWorkspace* w) {
  if (sh.B < 1 || sh.S < 1 || sh.N < 1) return false;
  const int64_t tiles = (static_cast<int64_t>(sh.N) + dsa::kKeysPerTile - 1) / dsa::kKeysPerTile;
  const int64_t sample_tiles = (tiles + dsa::kSampleEvery - 1) / dsa::kSampleEvery;
  const int64_t filtered_tiles = tiles - sample_tiles;
  w->rows = static_cast<int64_t>(sh.B) * sh.S;
  w->ns_cols = sample_tiles * dsa::kKeysPerTile;
  w->cap = filtered_tiles * dsa::kKeysPerTile;
  w->mask_stride = filtered_tiles * 4;
  w->off_mask = 0;
  w->off_thr = align256(w->off_mask + 4 * w->mask_stride * w->rows);
  w->off_s = align256(w->off_thr + 4 * w->rows);
  w->off_c = align256(w->off_s + 4 * w->rows * w->ns_cols);
  w->bytes = align256(w->off_c + 4 * w->rows * w->cap);
  return true;
}

}  // namespace

extern "C" {

int64_t indexer_logits_topk_workspace_bytes(const idx_shape* shape) {
  TopkWorkspace w;
  if (shape == nullptr || !topk_workspace(*shape, &w)) return -1;
  return w.bytes;
}

int indexer_logits_topk(const void* q, const uint8_t* q_sf, const void* k, const uint8_t* k_sf,
                        const float* k_scales, const void* w, const int32_t* ks,
                        const int32_t* ke, float sm_scale, const idx_shape* shape, int32_t topk,
                        int32_t* idx, int64_t idx_stride, void* workspace,
                        int64_t workspace_bytes, idx_stream_t stream_) {
  if (!shape || !idx || !workspace) return IDX_ERR_NULL;
  if ((shape->flags & IDX_FLAG_OUT_BF16) != 0) return IDX_ERR_UNSUPPORTED;
  if (topk < 1 || idx_stride < topk) return IDX_ERR_SHAPE;
  TopkWorkspace ws;
  if (!topk_workspace(*shape, &ws)) return IDX_ERR_SHAPE;
  if (ws.rows > 0x7fffffffLL) return IDX_ERR_SHAPE;
  if (workspace_bytes < ws.bytes) return IDX_ERR_SCRATCH;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) || (reinterpret_cast<uintptr_t>(idx) & 3u))
    return IDX_ERR_ALIGN;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  char* base = static_cast<char*>(workspace);
  uint32_t* mask = reinterpret_cast<uint32_t*>(base + ws.off_mask);
  float* thr = reinterpret_cast<float*>(base + ws.off_thr);
  float* smp = reinterpret_cast<float*>(base + ws.off_s);
  float* kept = reinterpret_cast<float*>(base + ws.off_c);
  int sms = 0;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo* di = nullptr;
    int st = get_device_info(dev, &di);
    if (st) return st;
    sms = di->sm_count;
  }
  // The filter pass's mask words start at zero (cleared first, so that the
  // threshold and merge kernels directly follow the logits passes they read
  // and are launched as their programmatic dependents).
  if (cudaMemsetAsync(mask, 0, 4 * ws.mask_stride * ws.rows, stream) != cudaSuccess)
    return IDX_ERR_CUDA;
  // 1. the sample pass: every kSampleEvery-th key tile, compact FP32 rows
  PassArgs pass;
  pass.mode = dsa::kModeSample;
  pass.out_row_stride = ws.ns_cols;
  int st = enqueue_logits(q, q_sf, k, k_sf, k_scales, w, ks, ke, sm_scale, 1, smp, shape, stream,
                          false, nullptr, pass);
  if (st) return st;
  // 2. each row's threshold: the topk-th largest of its sample
  const unsigned grid = static_cast<unsigned>(ws.rows);
  const bool few = ws.rows <= 2LL * sms;
  constexpr int kMany = dsa::kTopkThreads, kFew = dsa::kTopkThreadsFew;
  const int ns = static_cast<int>(ws.ns_cols);
  st = few ? launch_dependent(dsa::topk_threshold_kernel<kFew>, grid, kFew, stream, smp,
                              ws.ns_cols, ns, topk, thr)
           : launch_dependent(dsa::topk_threshold_kernel<kMany>, grid, kMany, stream, smp,
                              ws.ns_cols, ns, topk, thr);
  if (st) return st;
  // 3. the other key tiles: append the values at or above the threshold
  pass.mode = dsa::kModeFilter;
  pass.out_row_stride = ws.cap;
  pass.thr = thr;
  pass.mask = mask;
  pass.mask_row_stride = ws.mask_stride;
  pass.planned = true;  // a grouped call's row order is the sample pass's
  if ((st = enqueue_logits(q, q_sf, k, k_sf, k_scales, w, ks, ke, sm_scale, 1, kept, shape, stream,
                           false, nullptr, pass)))
    return st;
  // 4. the top-k of sample and candidates
  return few ? launch_dependent(dsa::topk_merge_kernel<kFew>, grid, kFew, stream, smp, ws.ns_cols,
                                ns, kept, ws.cap, mask, ws.mask_stride, dsa::kSampleEvery, topk,
                                idx, idx_stride)
             : launch_dependent(dsa::topk_merge_kernel<kMany>, grid, kMany, stream, smp,
                                ws.ns_cols, ns, kept, ws.cap, mask, ws.mask_stride,
                                dsa::kSampleEvery, topk, idx, idx_stride);
}

int indexer_thd_windows(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                        int32_t num_seqs, int32_t total_q, int32_t causal, int32_t* ks,
                        int32_t* ke, idx_stream_t stream_) {
  if (!cu_seqlens_q || !cu_seqlens_k || !ks || !ke) return IDX_ERR_NULL;
  if (num_seqs < 1 || total_q < 1) return IDX_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) | reinterpret_cast<uintptr_t>(cu_seqlens_k) |
       reinterpret_cast<uintptr_t>(ks) | reinterpret_cast<uintptr_t>(ke)) & 3u)
    return IDX_ERR_ALIGN;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const unsigned blocks = static_cast<unsigned>((total_q + dsa::kWindowThreads - 1) / dsa::kWindowThreads);
  dsa::thd_windows_kernel<<<blocks, dsa::kWindowThreads, 0, stream>>>(
      cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, causal != 0, ks, ke);
  return cudaGetLastError() == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

int indexer_selftest_wait_timeout(int64_t limit_ns, idx_stream_t stream_) {
  if (limit_ns < 1000 || limit_ns > 1000000000LL) return IDX_ERR_SHAPE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ERR_CUDA;
  int32_t* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo* di = nullptr;
    int st = get_device_info(dev, &di);
    if (st) return st;
    if (di->cc_major != 10 || di->cc_minor != 3) return IDX_ERR_DEVICE;
    if ((st = get_scratch(dev, stream, kScratchInts, &scratch))) return st;
  }
  dsa::wait_selftest_kernel<<<1, 32, 0, stream>>>(scratch, static_cast<uint64_t>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

int indexer_noalloc_selftest_wait_timeout(int64_t limit_ns, idx_stream_t stream_) {
  if (limit_ns < 1000 || limit_ns > 1000000000LL) return IDX_ERR_SHAPE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ERR_CUDA;
  int32_t* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo* di = nullptr;
    int st = get_device_info(dev, &di);
    if (st) return st;
    if (di->cc_major != 10 || di->cc_minor != 3) return IDX_ERR_DEVICE;
    if ((st = get_fixed_scratch(dev, &scratch))) return st;
  }
  dsa::wait_selftest_kernel<<<1, 32, 0, stream>>>(scratch, static_cast<uint64_t>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

int indexer_shutdown(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int rc = IDX_OK;
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : g_scratch) {
    if (kv.second.ptr == nullptr) continue;
    if (cudaSetDevice(kv.first.first) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
        cudaFree(kv.second.ptr) != cudaSuccess)
      rc = IDX_ERR_CUDA;
  }
  g_scratch.clear();
  cudaSetDevice(cur);
  return rc;
}

}  // extern "C"
