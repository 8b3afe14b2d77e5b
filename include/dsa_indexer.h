/*
 * dsa_indexer.h — C ABI of the GB300 (sm_103a) lightning-indexer library.
 *
 * The operation (one call = one pass of the indexer's MQA-logits forward):
 *
 *   out[b,i,j] = sum_h w[b,i,h] * ReLU(sm_scale * q[b,i,h,:] . k[b,j,:])
 *                                              for ks[b,i] <= j < ke[b,i]
 *   out[b,i,j] = -inf                          for every other j < N (clean != 0)
 *
 * H query heads share one key head of dimension D. Defined by:
 *  - DeepGEMM pull request 435, "Improve SM100 MX MQA logits clean-output
 *    performance": the fp8_fp4_mqa_logits call in its "Standalone performance
 *    reproducer" section — (q, q_scales), (k, k_scales), weights, starts,
 *    ends, clean_logits, FP32 logits; windows [0, KV-Q+row) in "Performance";
 *    MX scales packed four E8M0 bytes per 32-bit word, 0x7f7f7f7f = all ones;
 *    -inf outside the window and 0 in-window for all-zero inputs.
 *  - cuDNN-frontend pull request 416, "DSA indexer forward: add a lean SM100
 *    fast path ...", sections "What", "Precision / determinism" and "Support
 *    surface": BF16 Q/K, BF16 or FP32 W, FP32 scores, H=64, D=128, h_kv=1,
 *    batched uniform-length BSHD, -inf outside the window, S_q % 4 == 0,
 *    16-byte aligned base pointers, finite sm_scale.
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument of a compute call is a DEVICE pointer on the
 *    current CUDA device, owned by the caller; the library never frees it.
 *  - Calls are asynchronous and ordered on `stream` (NULL = legacy default
 *    stream). They never synchronise and never read device data on the host.
 *  - A non-zero return is an idx_status; nothing was launched in that case.
 */
#ifndef DSA_INDEXER_H_
#define DSA_INDEXER_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define IDX_API __attribute__((visibility("default")))
#else
#define IDX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* idx_stream_t; /* same type as cudaStream_t */

/* Element format of Q and K (both use the same one). */
typedef enum idx_format {
  IDX_FMT_BF16 = 0,  /* bfloat16 elements; D elements per row                 */
  IDX_FMT_E4M3 = 1,  /* OCP FP8 E4M3; optional FP32 per-key scale (k_scales)   */
  IDX_FMT_MXFP8 = 2, /* E4M3 + one E8M0 scale per 32 elements of D            */
  IDX_FMT_MXFP4 = 3  /* E2M1, two per byte (even element in the low nibble),
                        + one E8M0 scale per 32 elements of D                  */
} idx_format;

/* Element format of the head weights w. */
typedef enum idx_w_format { IDX_W_F32 = 0, IDX_W_BF16 = 1 } idx_w_format;

typedef enum idx_status {
  IDX_OK = 0,
  IDX_ERR_NULL = 1,        /* a required pointer is NULL                            */
  IDX_ERR_SHAPE = 2,       /* H != 64, D != 128, B/S/N < 1, out_row_stride < N, or a
                              size beyond int32 indexing                              */
  IDX_ERR_FORMAT = 3,      /* unknown fmt / w_fmt, or scales missing for MX          */
  IDX_ERR_ALIGN = 4,       /* q/k/w base or q/k stride not 16-byte aligned, or out
                              not aligned to its element size                         */
  IDX_ERR_SCALE = 5,       /* sm_scale is not finite                                  */
  IDX_ERR_DEVICE = 6,      /* current device is not compute capability 10.3 (sm_103) */
  IDX_ERR_CUDA = 7,        /* a CUDA runtime call failed (launch, allocation, ...)   */
  IDX_ERR_TIMEOUT = 8,     /* device-side wait gave up; the call's output is invalid */
  IDX_ERR_UNSUPPORTED = 9, /* valid request this build does not implement            */
  IDX_ERR_SCRATCH = 10     /* indexer_logits_noalloc: more scratch than its array;
                              indexer_logits_topk: workspace too small               */
} idx_status;

/* idx_shape.flags: the rows' windows are irregular (not a causal staircase);
 * group rows with similar windows into the kernel's 4-row blocks. A block
 * computes the union of its rows' 128-key tiles, so on windows with unrelated
 * starts and lengths consecutive rows waste about 2.4x the work; grouped, about
 * 1.03x. Costs one extra launch (a per-batch counting sort of the rows by
 * window) and B*S*4 bytes of library scratch on the stream; ignored by
 * indexer_logits_noalloc. The logits do not depend on it (nor on the order
 * of rows inside a bin, which may differ between calls). */
#define IDX_FLAG_GROUP_ROWS 1

/* idx_shape.flags: write the logits as BF16 (round to nearest even of the
 * FP32 result; -inf stays -inf) instead of FP32, halving the bytes stored.
 * The output then holds BF16 elements and out_row_stride counts BF16
 * elements. DeepGEMM's MX logits call takes the same choice as its
 * logits_dtype argument. */
#define IDX_FLAG_OUT_BF16 2

/* Problem shape and layout. Zero strides mean "dense". */
typedef struct idx_shape {
  int32_t B;              /* batches (uniform length), >= 1                          */
  int32_t S;              /* query rows per batch, >= 1                               */
  int32_t N;              /* keys per batch, >= 1                                      */
  int32_t H;              /* query heads, must be 64                                   */
  int32_t D;              /* head dimension, must be 128                               */
  int32_t fmt;            /* idx_format                                                */
  int32_t w_fmt;          /* idx_w_format                                              */
  int32_t flags;          /* IDX_FLAG_* bits, other bits 0                             */
  int64_t q_row_bytes;    /* bytes between consecutive (b,i,h) rows of q; 0 = dense    */
  int64_t k_row_bytes;    /* bytes between consecutive keys of k; 0 = dense            */
  int64_t k_batch_bytes;  /* bytes between batches of k; 0 = N * k_row_bytes           */
  int64_t out_row_stride; /* elements between consecutive output rows; 0 = N           */
} idx_shape;

/* Compute the logits (one call of the hot path).
 *
 *  q        [B,S,H,D] elements (MXFP4: D/2 bytes per (b,i,h) row), row stride
 *           q_row_bytes (multiple of 16), base 16-byte aligned; batches and
 *           rows contiguous at that stride.
 *  q_sf     MX formats: E8M0 bytes [B,S,H,D/32], dense (byte g of a head row
 *           scales elements 32g..32g+31; the four bytes of a row read as a
 *           little-endian int32 are DeepGEMM's packed q_scales); else NULL.
 *  k        [B,N,D] elements (MXFP4: D/2 bytes per key), strides k_row_bytes
 *           and k_batch_bytes (multiples of 16), base 16-byte aligned.
 *  k_sf     MX formats: E8M0 bytes [B,N,D/32], dense; else NULL.
 *  k_scales IDX_FMT_E4M3 only: FP32 [B,N] per-key scale >= 0 multiplying K
 *           (a per-query-row Q scale belongs in w); NULL means 1. Must be NULL
 *           for the other formats.
 *  w        [B,S,H] FP32 or BF16 (w_fmt), dense, base 16-byte aligned.
 *  ks, ke   [B,S] int32, dense. Row (b,i) sees keys [max(ks,0), min(ke,N));
 *           ks >= ke is an empty row (all -inf). Values are clamped on the
 *           device; any int32 is accepted.
 *  sm_scale finite float; it multiplies the dot product inside the ReLU (a
 *           negative value is honoured exactly: ReLU(s*x) = |s|*ReLU(-x)).
 *  clean    non-zero: every column j < N outside the window is written -inf.
 *           zero: columns of 128-key tiles that contain no in-window key of
 *           any row of the row's block (4 rows; 2 where every batch has at
 *           most two rows and the keys are BF16 or E4M3) are left untouched;
 *           the rest is written (-inf outside the window).
 *  out      FP32 (BF16 with IDX_FLAG_OUT_BF16) [B,S,out_row_stride], base
 *           aligned to its element size; columns >= N are never written.
 *  shape    see idx_shape (host pointer, read during the call only).
 *  stream   CUDA stream of the launch.
 *
 * Returns IDX_OK once the work is enqueued. Argument errors are detected on
 * the host before any launch. A device-side wait that runs out is reported
 * by indexer_get_last_error(), not here. The first call on a (device,
 * stream) pair allocates a small library-owned scratch block (a work counter
 * and an error word, plus B*S words for IDX_FLAG_GROUP_ROWS, plus for the MX
 * formats 512 bytes per (batch, 128-key tile) holding the key scale words in
 * the kernel's copy order) from the device's stream-ordered pool; a later call that needs more grows it on `stream`
 * (cudaMallocAsync / cudaFreeAsync, no synchronisation). Make one call of the
 * largest shape before capturing a CUDA graph on that stream, and release a
 * short-lived stream's block with indexer_stream_release;
 * calls on one stream reuse it, so calls on the same stream must not overlap
 * (stream order guarantees that).
 */
IDX_API int indexer_logits(const void* q, const uint8_t* q_sf, const void* k, const uint8_t* k_sf,
                   const float* k_scales, const void* w, const int32_t* ks, const int32_t* ke,
                   float sm_scale, int clean, void* out, const idx_shape* shape,
                   idx_stream_t stream);

/* Same computation, arguments and checks as indexer_logits, but this call
 * never allocates device memory, not even on its first use. The pages have no
 * counterpart; it is here for callers that may not call cudaMalloc: code
 * running while a stream is being captured into a CUDA graph, allocators and
 * memory-pool owners, and embedders whose memory budget is fixed up front.
 *
 * Its scratch (a work counter, a finished-block count and an error word: 3 of
 * 64 words) lives in one fixed 256-byte device array inside the library, which
 * every GPU that loads the library keeps until the process exits. One call
 * needs the same 3 words whatever its shape, so no shape is turned away for
 * lack of scratch; IDX_ERR_SCRATCH is returned if a call would need more than
 * the array holds. The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, no allocation); make that first call before
 * any stream capture. Each call clears the three words on `stream` before its
 * kernel, because the array keeps the previous call's contents. All calls on
 * a device share the one array, so calls that can overlap on the GPU (on
 * different streams without ordering) race and must not be issued that way.
 * A device-side wait that runs out is recorded in that shared array, not in
 * the per-stream word indexer_get_last_error reads: read it with
 * indexer_noalloc_get_last_error after the call and before the next
 * no-allocation call on the device (which clears it). With no scratch for the
 * MX key scale words in copy order, an MX call here launches no pre-pass: its
 * kernel copies each key's scale word itself (measured 3-4% slower on MXFP8). */
IDX_API int indexer_logits_noalloc(const void* q, const uint8_t* q_sf, const void* k,
                                   const uint8_t* k_sf, const float* k_scales, const void* w,
                                   const int32_t* ks, const int32_t* ke, float sm_scale,
                                   int clean, void* out, const idx_shape* shape,
                                   idx_stream_t stream);

/* Keys in a paged cache (decode-time KV caches): key j of batch b is row
 * j % page_size of page block_table[b * table_stride + j / page_size]. The
 * pages need not be contiguous or in order, and batches may share pages. */
typedef struct idx_paged {
  const int32_t* block_table; /* device, [B, table_stride] int32 page numbers; entries
                                 for keys < N must lie in [0, num_pages) (others are
                                 clamped on the device: wrong values, no fault)      */
  int32_t table_stride;       /* entries per batch, >= ceil(N / page_size)             */
  int32_t page_size;          /* keys per page, a positive multiple of 64              */
  int32_t num_pages;          /* pages in the cache; num_pages * page_size < 2^31      */
  int32_t reserved;           /* must be 0                                             */
} idx_paged;

/* indexer_logits with the keys in a paged cache (no counterpart signature on
 * the pages, which only name DeepGEMM's paged MQA-logits path and its
 * tests). Arguments as for indexer_logits except:
 *  k_cache        [num_pages, page_size, D] elements (MXFP4: D/2 bytes per
 *                 key), row stride shape->k_row_bytes (0 = dense), base
 *                 16-byte aligned; shape->k_batch_bytes must be 0.
 *  k_sf_cache     MX formats: E8M0 [num_pages, page_size, D/32]; else NULL.
 *  k_scales_cache IDX_FMT_E4M3: FP32 [num_pages, page_size] per-key scales or
 *                 NULL; NULL for the other formats.
 *  shape->N       keys per batch seen through the table (the longest
 *                 context); each row's window [ks, ke) selects its keys, e.g.
 *                 [0, context_len - next_n + t + 1) for decode token t.
 *  paged          host pointer, read during the call only.
 * Returns IDX_ERR_NULL for a NULL paged/block_table, IDX_ERR_SHAPE for a bad
 * page size, table stride, page count or a non-zero k_batch_bytes; otherwise
 * as indexer_logits. The logits equal those of indexer_logits on the keys
 * gathered into a contiguous [B, N] array, bit for bit. */
IDX_API int indexer_paged_logits(const void* q, const uint8_t* q_sf, const void* k_cache,
                                 const uint8_t* k_sf_cache, const float* k_scales_cache,
                                 const void* w, const int32_t* ks, const int32_t* ke,
                                 float sm_scale, int clean, void* out, const idx_shape* shape,
                                 const idx_paged* paged, idx_stream_t stream);

/* Top-k selection over logits (DeepSeek Sparse Attention keeps each query's
 * top-2048 keys; the pages name it as the indexer's consumer): for every row,
 * the column indices of its k largest finite values. -inf (outside the row's
 * window) is never selected; a row with fewer than k finite values gets all
 * of them and -1 in the rest of its k slots. Indices come out in no
 * particular order; among values equal to the k-th largest, any subset of
 * the right size is taken (the choice may differ between calls).
 *  logits       device, [rows, row_stride] FP32, or BF16 when logits_bf16 is
 *               non-zero (the output of indexer_logits with either format);
 *               base aligned to the element size.
 *  rows, N      rows >= 1 (at most 2^31 - 1), columns N >= 1, N <= row_stride.
 *  k            1 <= k.
 *  idx          device, [rows, idx_stride] int32, idx_stride >= k; written in
 *               columns [0, k) of every row.
 * Stream-ordered like every call: the selection kernel is launched as a
 * programmatic dependent of the previous kernel on `stream`, so it may be
 * placed on the GPU while that kernel finishes, but it reads the logits only
 * after that kernel has completed.
 * Returns IDX_OK once enqueued; IDX_ERR_NULL, IDX_ERR_SHAPE, IDX_ERR_ALIGN,
 * IDX_ERR_DEVICE, IDX_ERR_CUDA as for indexer_logits. */
IDX_API int indexer_topk(const void* logits, int logits_bf16, int64_t rows, int32_t N,
                         int64_t row_stride, int32_t k, int32_t* idx, int64_t idx_stride,
                         idx_stream_t stream);

/* Bytes of device workspace indexer_logits_topk needs for this shape (any
 * top-k size), or -1 for a NULL or invalid shape: about 4.1 * B*S*N bytes
 * (as much as the FP32 logits would take), i.e. per row 4 bytes for each key
 * (the sampled logits of one 128-key tile in four, a value slot for each key
 * of the other tiles, so that no input can overflow it) and a mask word per
 * 32 keys of the other tiles. Only kept values are written to the slots
 * (packed at the front of each 32-key group). */
IDX_API int64_t indexer_logits_topk_workspace_bytes(const idx_shape* shape);

/* The indexer's logits reduced straight to each row's top-k key columns, the
 * way DeepSeek Sparse Attention consumes them (the FlashInfer page's sparse
 * MLA prefill takes top-k = 2048 indices per query), without writing the
 * B*S*N logits. Same inputs, checks and windows as indexer_logits (shape
 * flags: IDX_FLAG_GROUP_ROWS only; clean is implied), and the same result as
 * indexer_topk over indexer_logits' FP32 output: for every row the columns of
 * its `topk` largest in-window logits, in no particular order, -1 padding
 * when the window holds fewer; among values equal to the topk-th largest any
 * subset of the right size. The logits are computed exactly as
 * indexer_logits computes them.
 *
 * How: a first pass computes the logits of every fourth 128-key tile into
 * the workspace; the topk-th largest of them is a lower bound T of the row's
 * topk-th largest logit (those topk values are logits of the row); a second
 * pass over the other tiles keeps only in-window logits >= T (packed per 32
 * keys in the workspace, with a bit mask per 32 keys); a last selection
 * takes the top-k of the sampled logits and the kept values. Five launches on `stream` (six with
 * IDX_FLAG_GROUP_ROWS), no synchronisation, no host read of device data.
 *
 *  topk       >= 1.
 *  idx        device, int32 [B*S, idx_stride], idx_stride >= topk; row b*S+i
 *             gets its columns in [0, topk).
 *  workspace  device, 256-byte aligned, at least
 *             indexer_logits_topk_workspace_bytes(shape) bytes, owned by the
 *             caller; its contents are scratch (not kept between calls).
 * Returns IDX_ERR_SCRATCH if workspace_bytes is too small,
 * IDX_ERR_UNSUPPORTED for IDX_FLAG_OUT_BF16, otherwise as indexer_logits.
 * Contiguous keys only (no paged variant). */
IDX_API int indexer_logits_topk(const void* q, const uint8_t* q_sf, const void* k,
                                const uint8_t* k_sf, const float* k_scales, const void* w,
                                const int32_t* ks, const int32_t* ke, float sm_scale,
                                const idx_shape* shape, int32_t topk, int32_t* idx,
                                int64_t idx_stride, void* workspace, int64_t workspace_bytes,
                                idx_stream_t stream);

/* Windows of sequences packed along the rows and keys of one batch (the
 * THD / varlen layout: cuDNN-frontend pull request 416, "What" and its THD
 * commit), computed on the device from cumulative lengths, for a call with
 * B = 1, S = total_q and N = the packed key count; its logits columns are
 * then global key positions.
 *  cu_seqlens_q, cu_seqlens_k  device int32 [num_seqs + 1], non-decreasing,
 *               starting at 0: sequence s owns rows [cu_q[s], cu_q[s+1]) and
 *               keys [cu_k[s], cu_k[s+1]).
 *  causal       non-zero: row r of a sequence with n_q rows and n_k keys sees
 *               its first clamp(n_k - n_q + r + 1, 0, n_k) keys (the last row
 *               all of them); zero: all n_k keys.
 *  ks, ke       device int32 [total_q] written with absolute windows; rows at
 *               or past cu_q[num_seqs] get the empty window [0, 0).
 * Asynchronous on `stream`; IDX_ERR_NULL, IDX_ERR_SHAPE (num_seqs or total_q
 * < 1), IDX_ERR_ALIGN (pointers not 4-byte aligned), IDX_ERR_CUDA. */
IDX_API int indexer_thd_windows(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                int32_t num_seqs, int32_t total_q, int32_t causal, int32_t* ks,
                                int32_t* ke, idx_stream_t stream);

/* Human-readable text for an idx_status value (static storage, never NULL). */
IDX_API const char* indexer_status_string(int status);

/* Synchronise `stream`, then return and clear the device-side error word of
 * that (current device, stream) pair: IDX_OK, or IDX_ERR_TIMEOUT if a kernel
 * on it gave up waiting (its output is then invalid). Returns IDX_OK when no
 * call was ever made on the pair, IDX_ERR_CUDA if synchronisation fails. */
IDX_API int indexer_get_last_error(idx_stream_t stream);

/* indexer_get_last_error for indexer_logits_noalloc: synchronise `stream`,
 * then return and clear the error word of the current device's fixed
 * no-allocation array (IDX_OK, or IDX_ERR_TIMEOUT if the last no-allocation
 * call on the device gave up waiting; its output is then invalid). Call it
 * before the next no-allocation call on the device, which clears the word.
 * Allocates nothing. Returns IDX_OK when no no-allocation call was ever made
 * on the device, IDX_ERR_CUDA if synchronisation fails. */
IDX_API int indexer_noalloc_get_last_error(idx_stream_t stream);

/* Free the library scratch block of the (current device, stream) pair, if
 * any, stream-ordered on `stream` (no synchronisation). A caller that makes
 * calls on short-lived streams calls this after its last call on a stream and
 * before destroying it; otherwise each such stream keeps its block (256 bytes,
 * plus B*S words after grouped calls) until indexer_shutdown. A later call on
 * the pair allocates again. Returns IDX_OK or IDX_ERR_CUDA. */
IDX_API int indexer_stream_release(idx_stream_t stream);

/* Device-side wait limit in nanoseconds for later launches from this process
 * (default 2e9). Used by tests to make a wait run out on purpose; values
 * below 1e6 are raised to 1e6. Returns the previous value. */
IDX_API int64_t indexer_set_wait_limit_ns(int64_t ns);

/* Failure-detection self-test (no counterpart in the method: a diagnostic
 * of this library). Enqueues on `stream` one device-side wait of the kind the
 * logits kernel's roles use, on a barrier that nothing arrives on, so that it
 * runs out after `limit_ns` nanoseconds (1e3 .. 1e9, else IDX_ERR_SHAPE) and
 * records IDX_ERR_TIMEOUT in the (device, stream) error word, as a logits call
 * that gave up would; indexer_get_last_error(stream) then returns
 * IDX_ERR_TIMEOUT and clears it. Nothing else is in flight, so the context
 * stays usable. Returns IDX_OK once enqueued, IDX_ERR_DEVICE off sm_103,
 * IDX_ERR_CUDA if allocation or launch fails. */
IDX_API int indexer_selftest_wait_timeout(int64_t limit_ns, idx_stream_t stream);

/* The failure-detection self-test above, aimed at the fixed array of
 * indexer_logits_noalloc instead of a per-stream word (no counterpart in the
 * method; allocates nothing): indexer_noalloc_get_last_error then returns
 * IDX_ERR_TIMEOUT once and clears it. Same limits and returns as
 * indexer_selftest_wait_timeout. */
IDX_API int indexer_noalloc_selftest_wait_timeout(int64_t limit_ns, idx_stream_t stream);

/* Number of kernel launches one indexer_logits (or indexer_paged_logits)
 * call with this shape makes: the logits kernel, plus one with
 * IDX_FLAG_GROUP_ROWS in effect (the row order) and one for the MX formats
 * (their key scale words put in the kernel's copy order);
 * indexer_logits_noalloc makes neither extra launch. For launch counts in
 * benchmarks. */
IDX_API int indexer_launches_per_call(const idx_shape* shape);

/* Free every library-owned scratch block on every device (synchronises each
 * device that has one). Later calls allocate again. Returns IDX_OK or
 * IDX_ERR_CUDA. */
IDX_API int indexer_shutdown(void);

/* Library ABI version: major*10000 + minor*100 + patch. */
IDX_API int indexer_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_INDEXER_H_ */
