/*
 * Float64 CPU oracle for the DeepSeek-Sparse-Attention "lightning indexer"
 * MQA-logits forward.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
 * call this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do. It shares no code, header, table or constant with the
 * CUDA library: it has its own element decoders, written from the format
 * definitions, and it works on the raw input bytes.
 *
 * What it computes (one plain loop nest, no blocking, no reordering):
 *
 *   logits[b,i,j] = sum_h w[b,i,h] * max(0, sm_scale * sum_d Qd[b,i,h,d] * Kd[b,j,d])
 *                                                   for lo_i <= j < hi_i
 *   logits[b,i,j] = -inf                            otherwise
 *
 *   lo_i = max(ks[b,i], 0), hi_i = min(ke[b,i], N); lo_i >= hi_i is an empty row.
 *
 * Sources:
 *  - The formula, the half-open window [ks, ke), the -inf fill of every column
 *    outside it and one K head shared by all H query heads: DeepGEMM pull
 *    request 435, "Improve SM100 MX MQA logits clean-output performance",
 *    sections "Performance" (window [0, KV-Q+row)) and "Standalone performance
 *    reproducer" (the fp8_fp4_mqa_logits call with starts/ends and
 *    clean_logits, and its check that the -inf pattern is exactly the
 *    complement of cols < ends with zeros in-window for all-zero inputs).
 *  - FP32 scores, -inf outside the causal window, BF16 Q/K with BF16 or FP32
 *    W: cuDNN-frontend pull request 416, "DSA indexer forward: add a lean
 *    SM100 fast path ...", sections "What" and "Precision / determinism".
 *  - Element formats: OCP Microscaling (MX) Formats specification v1.0
 *    (E4M3, E2M1 element encodings; E8M0 shared scale = 2^(e-127), 0xFF NaN;
 *    one scale per 32-element block), and the bfloat16 format (IEEE binary32
 *    with the low 16 mantissa bits removed).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - ks is inclusive, ke exclusive; out-of-range values are clamped to
 *    [0, N]; ks >= ke gives an all -inf row.
 *  - sm_scale multiplies the dot product inside the ReLU.
 *  - FP8 per-token: Kd[b,j,d] = e4m3(K[b,j,d]) * k_scale[b,j]. The per-row Q
 *    scale is already folded into W by whoever made the inputs.
 *  - MX: Xd = element * 2^(E8M0 - 127), the scale of block d/32 of that row
 *    (and head, for Q). FP4 packs two elements per byte, low nibble = even d.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_E4M3 = 1, ORC_MXFP8 = 2, ORC_MXFP4 = 3 };
enum { ORC_W_F32 = 0, ORC_W_BF16 = 1 };

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 mantissa bits. */
double orc_decode_bf16(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 7) & 0xFF;
  int m = bits & 0x7F;
  double v;
  if (e == 0xFF) {
    v = (m == 0) ? INFINITY : NAN;
  } else if (e == 0) {
    v = ldexp((double)m / 128.0, -126);
  } else {
    v = ldexp(1.0 + (double)m / 128.0, e - 127);
  }
  return sign ? -v : v;
}

/* OCP E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinity;
 * S.1111.111 is NaN; max normal 448; subnormals m/8 * 2^-6. */
double orc_decode_e4m3(uint8_t bits) {
  int sign = (bits >> 7) & 1;
  int e = (bits >> 3) & 0xF;
  int m = bits & 0x7;
  double v;
  if (e == 0xF && m == 0x7) {
    v = NAN;
  } else if (e == 0) {
    v = ldexp((double)m / 8.0, -6);
  } else {
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  }
  return sign ? -v : v;
}

/* OCP E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; no inf/NaN.
 * Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_decode_e2m1(uint8_t nibble) {
  int sign = (nibble >> 3) & 1;
  int e = (nibble >> 1) & 0x3;
  int m = nibble & 0x1;
  double v;
  if (e == 0) {
    v = (double)m * 0.5;
  } else {
    v = ldexp(1.0 + (double)m / 2.0, e - 1);
  }
  return sign ? -v : v;
}

/* OCP E8M0 shared scale: 2^(bits - 127); 0xFF is NaN. */
double orc_decode_e8m0(uint8_t bits) {
  if (bits == 0xFF) return NAN;
  return ldexp(1.0, (int)bits - 127);
}

/* Dequantise one row of D elements of a Q head or a K key.
 *   data   : the row's first byte (FP4: D/2 bytes, else D elements)
 *   sf     : the row's D/32 E8M0 bytes (MX formats), else unused
 *   extra  : per-token multiplier (FP8 per-token K scale), 1.0 otherwise */
static void dequant_row(int fmt, const uint8_t* data, const uint8_t* sf, int D,
                        double extra, double* dst) {
  for (int d = 0; d < D; ++d) {
    double x;
    switch (fmt) {
      case ORC_BF16: {
        uint16_t bits;
        memcpy(&bits, data + 2 * (size_t)d, 2);
        x = orc_decode_bf16(bits);
        break;
      }
      case ORC_E4M3:
        x = orc_decode_e4m3(data[d]);
        break;
      case ORC_MXFP8:
        x = orc_decode_e4m3(data[d]) * orc_decode_e8m0(sf[d / 32]);
        break;
      case ORC_MXFP4: {
        uint8_t byte = data[d / 2];
        uint8_t nib = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
        x = orc_decode_e2m1(nib) * orc_decode_e8m0(sf[d / 32]);
        break;
      }
      default:
        x = NAN;
    }
    dst[d] = x * extra;
  }
}

static size_t row_bytes(int fmt, int D) {
  switch (fmt) {
    case ORC_BF16: return 2 * (size_t)D;
    case ORC_MXFP4: return (size_t)D / 2;
    default: return (size_t)D;
  }
}

/*
 * Full oracle. All arrays are dense and row-major:
 *   q      [B,S,H, row_bytes(fmt,D)]     q_sf [B,S,H,D/32] (MX only)
 *   k      [B,N,   row_bytes(fmt,D)]     k_sf [B,N,D/32]   (MX only)
 *   k_tok  [B,N] float32 per-key scale (FP8 per-token) or NULL
 *   w      [B,S,H] float32 (w_fmt 0) or bfloat16 bits (w_fmt 1)
 *   ks, ke [B,S] int32
 *   rows   flattened row ids b*S+i to evaluate (NULL: all B*S rows, nrows ignored)
 *   out    [nrows, N] float64 logits, -inf outside the window
 *   den    [nrows, N] float64 sum_h |w|*|sm_scale*q_h.k| (or NULL); 0 outside
 *   den_abs[nrows, N] float64 sum_h |w|*|sm_scale|*sum_d |q_hd||k_d| (or NULL)
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int orc_logits(int fmt, int w_fmt, const void* q, const uint8_t* q_sf,
               const void* k, const uint8_t* k_sf, const float* k_tok,
               const void* w, const int32_t* ks, const int32_t* ke, int B,
               int S, int N, int H, int D, double sm_scale,
               const int64_t* rows, int64_t nrows, double* out, double* den,
               double* den_abs, int nthreads) {
  if (!q || !k || !w || !ks || !ke || !out) return -1;
  if (B < 1 || S < 0 || N < 0 || H < 1 || D < 1) return -1;
  if ((fmt == ORC_MXFP8 || fmt == ORC_MXFP4) && (D % 32 != 0 || !q_sf || !k_sf)) return -1;
  if (fmt < ORC_BF16 || fmt > ORC_MXFP4) return -1;
  if (rows == NULL) nrows = (int64_t)B * S;

  const size_t rb = row_bytes(fmt, D);
  const int nblk = D / 32;

  /* Dequantise every key once: Kd[b,j,:]. */
  double* kd = (double*)malloc(sizeof(double) * (size_t)B * (size_t)N * (size_t)D + 1);
  if (!kd) return -1;
  for (int64_t bj = 0; bj < (int64_t)B * N; ++bj) {
    const uint8_t* src = (const uint8_t*)k + (size_t)bj * rb;
    const uint8_t* sf = k_sf ? k_sf + (size_t)bj * nblk : NULL;
    double extra = k_tok ? (double)k_tok[bj] : 1.0;
    dequant_row(fmt, src, sf, D, extra, kd + (size_t)bj * D);
  }

  int status = 0;
#ifdef _OPENMP
  if (nthreads < 1) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t row = rows ? rows[r] : r;
    double* orow = out + (size_t)r * N;
    double* drow = den ? den + (size_t)r * N : NULL;
    double* arow = den_abs ? den_abs + (size_t)r * N : NULL;
    double* qd = (double*)malloc(sizeof(double) * (size_t)H * D);
    double* wd = (double*)malloc(sizeof(double) * (size_t)H);
    if (!qd || !wd || row < 0 || row >= (int64_t)B * S) {
      free(qd);
      free(wd);
#ifdef _OPENMP
#pragma omp atomic write
#endif
      status = -1;
      continue;
    }
    const int64_t b = row / S;
    for (int h = 0; h < H; ++h) {
      const size_t qh = (size_t)row * H + h;
      dequant_row(fmt, (const uint8_t*)q + qh * rb, q_sf ? q_sf + qh * nblk : NULL,
                  D, 1.0, qd + (size_t)h * D);
      if (w_fmt == ORC_W_BF16) {
        uint16_t bits;
        memcpy(&bits, (const uint8_t*)w + 2 * qh, 2);
        wd[h] = orc_decode_bf16(bits);
      } else {
        wd[h] = (double)((const float*)w)[qh];
      }
    }
    int64_t lo = ks[row] > 0 ? ks[row] : 0;
    int64_t hi = ke[row] < N ? ke[row] : N;
    for (int64_t j = 0; j < N; ++j) {
      if (j < lo || j >= hi) {
        orow[j] = -INFINITY;
        if (drow) drow[j] = 0.0;
        if (arow) arow[j] = 0.0;
        continue;
      }
      const double* kj = kd + ((size_t)b * N + (size_t)j) * D;
      double acc = 0.0, dn = 0.0, da = 0.0;
      for (int h = 0; h < H; ++h) {
        const double* qh = qd + (size_t)h * D;
        double dot = 0.0, dabs = 0.0;
        for (int d = 0; d < D; ++d) {
          dot += qh[d] * kj[d];
          dabs += fabs(qh[d]) * fabs(kj[d]);
        }
        double x = sm_scale * dot;
        acc += wd[h] * (x > 0.0 ? x : 0.0);
        dn += fabs(wd[h]) * fabs(x);
        da += fabs(wd[h]) * fabs(sm_scale) * dabs;
      }
      orow[j] = acc;
      if (drow) drow[j] = dn;
      if (arow) arow[j] = da;
    }
    free(qd);
    free(wd);
  }
  free(kd);
  return status;
}

/* Exported for the pins: dequantise one row (Q head or K key) of D elements. */
int orc_dequant_row(int fmt, const uint8_t* data, const uint8_t* sf, int D,
                    double extra, double* dst) {
  if (!data || !dst || D < 1) return -1;
  if ((fmt == ORC_MXFP8 || fmt == ORC_MXFP4) && (!sf || D % 32 != 0)) return -1;
  dequant_row(fmt, data, sf, D, extra, dst);
  return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
