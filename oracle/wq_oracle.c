/*
 * wq_oracle.c -- plain, slow, obviously-correct CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY: called by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  Single-threaded;
 * double accumulation (int64 for the W8A8 integer product); no blocking,
 * fusion or reordering beyond the loop order of a plain sum.
 *
 * Sources of the definitions (web pages, by title and section):
 *   [QC]  "Quantization CUDA" (tom-jerr.github.io)
 *         - Weight Only Quantization / 量化粒度: x = S * (q - Z), per-channel,
 *           per-token and group-wise granularity;
 *         - Int8 Weight Only Quantization: Y = (X . Wint) * Sw;
 *         - Dynamic Quantization: Y = Sx * (Xint . Wint) * Sw, int8 multiply,
 *           int32 accumulate, rescale to float;
 *         - Int4 Weight Only Quantization / Weight Store: int4 codes packed
 *           into a wider word, consecutive along K;
 *         - Marlin 格式: eight INT4 codes per INT32, W = (Wint4 - Zero) * Scale.
 *   [GK]  GPTQ CUDA kernel walkthrough (yelogs.com), section CUDA核函數設計與實現:
 *         3-bit codes extracted from int32 words with (word >> 3j) & 0x7 and
 *         dequantized as scale * q - zero.
 *   [FD]  "融合反量化与GEMM：LLM推理的CUDA内核优化实践" (zingnex.cn), section
 *         量化策略：分组对称INT8: symmetric INT8 with one scale per 128 elements.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - 3-bit codes that straddle a word boundary: the 32 codes of a block are
 *     one 96-bit little-endian bit stream (code 10 = bits 30..31 of word 0 and
 *     bit 0 of word 1; code 21 = bit 31 of word 1 and bits 0..1 of word 2);
 *   - 4-bit nibble j of a word holds row 8r + j; zero points are packed eight
 *     per int32 along N and stored without an offset;
 *   - W8A8: Sx = fp32(max|row| / 127), codes by fp32 division then
 *     round-half-even, clamped to [-127, 127]; an all-zero row has Sx = 0 and
 *     codes 0.
 */
#include "wq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Scalar formats, written from the IEEE 754 definitions.                   */
/* ------------------------------------------------------------------------ */

double wqo_f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
  return sign ? -v : v;
}

double wqo_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;              /* bf16 = top half of fp32 */
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round |a| (finite, > 0) to a binary format with `prec` significand bits and
 * minimum normal exponent `emin`; returns the rounded magnitude (exact in
 * double).  Ties go to even because nearbyint() runs in the default
 * round-to-nearest-even mode and a / quantum is exact. */
static double round_to_format(double a, int prec, int emin) {
  int e;
  frexp(a, &e);                  /* a = f * 2^e, f in [0.5, 1) */
  int lead = e - 1;              /* exponent of the leading bit */
  if (lead < emin) lead = emin;  /* subnormal range: fixed quantum */
  double quantum = ldexp(1.0, lead - (prec - 1));
  return nearbyint(a / quantum) * quantum;
}

uint16_t wqo_double_to_f16(double v) {
  if (isnan(v)) return 0x7e00;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  double r = round_to_format(a, 11, -14);
  if (r > 65504.0) return (uint16_t)(sign | 0x7c00);          /* overflow */
  if (r < ldexp(1.0, -14))                                      /* subnormal */
    return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -24)));
  int e;
  frexp(r, &e);
  int lead = e - 1;
  uint16_t mant = (uint16_t)(r / ldexp(1.0, lead - 10) - 1024.0);
  return (uint16_t)(sign | ((lead + 15) << 10) | mant);
}

uint16_t wqo_double_to_bf16(double v) {
  if (isnan(v)) return 0x7fc0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  double r = round_to_format(a, 8, -126);
  double maxv = ldexp(255.0, 127 - 7);                          /* (2 - 2^-7) * 2^127 */
  if (r > maxv) return (uint16_t)(sign | 0x7f80);
  if (r < ldexp(1.0, -126))
    return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -133)));
  int e;
  frexp(r, &e);
  int lead = e - 1;
  uint16_t mant = (uint16_t)(r / ldexp(1.0, lead - 7) - 128.0);
  return (uint16_t)(sign | ((lead + 127) << 7) | mant);
}

float wqo_double_to_f32(double v) { return (float)v; /* C: round to nearest even */ }

/* ------------------------------------------------------------------------ */
/* Code extraction.                                                         */
/* ------------------------------------------------------------------------ */

int wqo_code3(const int32_t* mat, int N, int k, int n) {
  /* [GK] CUDA核函數設計與實現: codes are read with (word >> 3j) & 7; the words
   * of one 32-code block are read as one little-endian bit stream. */
  int block = k / 32, j = k % 32;
  int bit = 3 * j;
  int word = bit / 32, off = bit % 32;
  uint32_t lo = (uint32_t)mat[(size_t)(3 * block + word) * N + n];
  uint32_t v = lo >> off;
  if (off > 29) { /* the code continues in the next word of the block */
    uint32_t hi = (uint32_t)mat[(size_t)(3 * block + word + 1) * N + n];
    v |= hi << (32 - off);
  }
  return (int)(v & 7u);
}

int wqo_code4(const int32_t* qweight, int N, int k, int n) {
  /* [QC] Int4 Weight Only Quantization / Weight Store and Marlin 格式:
   * eight 4-bit codes per 32-bit word, consecutive along K. */
  uint32_t word = (uint32_t)qweight[(size_t)(k / 8) * N + n];
  return (int)((word >> (4 * (k % 8))) & 15u);
}

int wqo_zero4(const int32_t* qzeros, int N, int g, int n) {
  uint32_t word = (uint32_t)qzeros[(size_t)g * (N / 8) + n / 8];
  return (int)((word >> (4 * (n % 8))) & 15u);
}

void wqo_unpack3(const int32_t* mat, int K, int N, uint8_t* codes) {
  for (int k = 0; k < K; ++k)
    for (int n = 0; n < N; ++n) codes[(size_t)k * N + n] = (uint8_t)wqo_code3(mat, N, k, n);
}

void wqo_unpack4(const int32_t* qweight, int K, int N, uint8_t* codes) {
  for (int k = 0; k < K; ++k)
    for (int n = 0; n < N; ++n) codes[(size_t)k * N + n] = (uint8_t)wqo_code4(qweight, N, k, n);
}

void wqo_unpack_zeros4(const int32_t* qzeros, int G, int N, uint8_t* zeros) {
  for (int g = 0; g < G; ++g)
    for (int n = 0; n < N; ++n) zeros[(size_t)g * N + n] = (uint8_t)wqo_zero4(qzeros, N, g, n);
}

/* ------------------------------------------------------------------------ */
/* The products.  For every requested column n and every row m:             */
/*   y[m,n] = sum_k x[m,k] * w(k,n)   accumulated in double, k ascending.   */
/* The loop runs k outermost so that each weight is decoded once and the    */
/* weight rows are read in memory order; the per-(m,n) sum is still the     */
/* plain ascending-k sum.                                                   */
/* ------------------------------------------------------------------------ */

static int col_of(const int32_t* cols, int c) { return cols ? cols[c] : c; }

void wqo_wq8_gemv(const float* x, const int8_t* w, const float* scales,
                  int M, int K, int N, int group,
                  const int32_t* cols, int ncols, double* y, double* abs_sum) {
  /* [QC] Int8 Weight Only Quantization: Y = X . (Wint * Sw);
   * [FD] 量化策略：分组对称INT8: one fp32 scale per group of 128 along K. */
  for (size_t i = 0; i < (size_t)M * ncols; ++i) { y[i] = 0.0; abs_sum[i] = 0.0; }
  for (int k = 0; k < K; ++k) {
    int g = k / group;
    for (int c = 0; c < ncols; ++c) {
      int n = col_of(cols, c);
      double wkn = (double)scales[(size_t)g * N + n] * (double)w[(size_t)k * N + n];
      for (int m = 0; m < M; ++m) {
        double t = (double)x[(size_t)m * K + k] * wkn;
        y[(size_t)m * ncols + c] += t;
        abs_sum[(size_t)m * ncols + c] += fabs(t);
      }
    }
  }
}

void wqo_wq3_gemv(const uint16_t* x, const int32_t* mat, const uint16_t* scales,
                  const uint16_t* zeros, int M, int K, int N,
                  const int32_t* cols, int ncols, double* y, double* abs_sum) {
  /* [GK] CUDA核函數設計與實現: res += (scale * q - zero) * vec[k]; the zero is
   * stored already multiplied by the scale. */
  for (size_t i = 0; i < (size_t)M * ncols; ++i) { y[i] = 0.0; abs_sum[i] = 0.0; }
  for (int k = 0; k < K; ++k) {
    for (int c = 0; c < ncols; ++c) {
      int n = col_of(cols, c);
      double s = wqo_f16_to_double(scales[n]);
      double zero = wqo_f16_to_double(zeros[n]);
      double wkn = s * (double)wqo_code3(mat, N, k, n) - zero;
      for (int m = 0; m < M; ++m) {
        double t = wqo_f16_to_double(x[(size_t)m * K + k]) * wkn;
        y[(size_t)m * ncols + c] += t;
        abs_sum[(size_t)m * ncols + c] += fabs(t);
      }
    }
  }
}

void wqo_wq4_gemm(const uint16_t* x, int act_bf16, const int32_t* qweight,
                  const uint16_t* scales, const int32_t* qzeros,
                  const int32_t* g_idx, int M, int K, int N, int group,
                  const int32_t* cols, int ncols, double* y, double* abs_sum) {
  /* [QC] 量化粒度 (group-wise): x = S * (q - Z) with one (S, Z) per group of
   * rows of one column; Marlin 格式: W = (Wint4 - Zero) * Scale.
   * Act-order: the group of row k is g_idx[k] instead of k / group. */
  double (*dec)(uint16_t) = act_bf16 ? wqo_bf16_to_double : wqo_f16_to_double;
  for (size_t i = 0; i < (size_t)M * ncols; ++i) { y[i] = 0.0; abs_sum[i] = 0.0; }
  for (int k = 0; k < K; ++k) {
    int g = g_idx ? g_idx[k] : k / group;
    for (int c = 0; c < ncols; ++c) {
      int n = col_of(cols, c);
      double s = dec(scales[(size_t)g * N + n]);
      int z = qzeros ? wqo_zero4(qzeros, N, g, n) : 8;
      double wkn = s * (double)(wqo_code4(qweight, N, k, n) - z);
      for (int m = 0; m < M; ++m) {
        double t = dec(x[(size_t)m * K + k]) * wkn;
        y[(size_t)m * ncols + c] += t;
        abs_sum[(size_t)m * ncols + c] += fabs(t);
      }
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Dequantization to a dense matrix (the separate-kernel path of            */
/* "融合反量化与GEMM", 核心优化思路: INT8 weights -> a dense buffer in DRAM ->  */
/* GEMM).  Each value is w(k,n) of the products above, exactly.             */
/* ------------------------------------------------------------------------ */

void wqo_wq8_dequant(const int8_t* w, const float* scales, int K, int N, int group, double* out) {
  for (int k = 0; k < K; ++k) {
    const float* srow = scales + (size_t)(k / group) * N;
    const int8_t* qrow = w + (size_t)k * N;
    for (int n = 0; n < N; ++n) out[(size_t)k * N + n] = (double)srow[n] * (double)qrow[n];
  }
}

void wqo_wq3_dequant(const int32_t* mat, const uint16_t* scales, const uint16_t* zeros,
                     int K, int N, double* out) {
  for (int k = 0; k < K; ++k)
    for (int n = 0; n < N; ++n) {
      double s = wqo_f16_to_double(scales[n]);
      out[(size_t)k * N + n] = s * (double)wqo_code3(mat, N, k, n) - wqo_f16_to_double(zeros[n]);
    }
}

void wqo_wq4_dequant(int act_bf16, const int32_t* qweight, const uint16_t* scales,
                     const int32_t* qzeros, const int32_t* g_idx, int K, int N, int group,
                     double* out) {
  double (*dec)(uint16_t) = act_bf16 ? wqo_bf16_to_double : wqo_f16_to_double;
  for (int k = 0; k < K; ++k) {
    int grp = g_idx ? g_idx[k] : k / group;
    for (int n = 0; n < N; ++n) {
      int zp = qzeros ? wqo_zero4(qzeros, N, grp, n) : 8;
      int q = wqo_code4(qweight, N, k, n);
      out[(size_t)k * N + n] = dec(scales[(size_t)grp * N + n]) * (double)(q - zp);
    }
  }
}

void wqo_w8a8_quant_rows(const uint16_t* X, int M, int K, int8_t* Xq, float* Sx) {
  /* [QC] Dynamic Quantization: activations are quantized at run time;
   * 量化粒度 (per-token): one scale per activation row. */
  for (int m = 0; m < M; ++m) {
    float amax = 0.0f;
    for (int k = 0; k < K; ++k) {
      float a = fabsf((float)wqo_bf16_to_double(X[(size_t)m * K + k]));
      if (a > amax) amax = a;
    }
    float sx = amax / 127.0f;                 /* fp32 division */
    Sx[m] = sx;
    for (int k = 0; k < K; ++k) {
      int q = 0;
      if (sx != 0.0f) {
        float r = (float)wqo_bf16_to_double(X[(size_t)m * K + k]) / sx;
        float rq = nearbyintf(r);             /* round half to even */
        if (rq > 127.0f) rq = 127.0f;
        if (rq < -127.0f) rq = -127.0f;
        q = (int)rq;
      }
      Xq[(size_t)m * K + k] = (int8_t)q;
    }
  }
}

void wqo_w8a8_quant_rows_smooth(const uint16_t* X, const float* smooth, int M, int K, int8_t* Xq,
                                float* Sx) {
  /* [QC] Smoothquant: Y = (X diag(s)^-1) . (diag(s) W): every activation is
   * divided by its channel's s (one correctly rounded fp32 division), then the
   * row is quantized exactly as in wqo_w8a8_quant_rows. */
  float* xs = (float*)malloc((size_t)K * sizeof(float));
  for (int m = 0; m < M; ++m) {
    float peak = 0.0f;
    for (int k = 0; k < K; ++k) {
      xs[k] = (float)wqo_bf16_to_double(X[(size_t)m * K + k]) / smooth[k];
      if (fabsf(xs[k]) > peak) peak = fabsf(xs[k]);
    }
    const float scale = peak / 127.0f;         /* fp32 division */
    Sx[m] = scale;
    for (int k = 0; k < K; ++k) {
      float code = 0.0f;
      if (scale != 0.0f) {
        code = nearbyintf(xs[k] / scale);      /* round half to even */
        code = code > 127.0f ? 127.0f : (code < -127.0f ? -127.0f : code);
      }
      Xq[(size_t)m * K + k] = (int8_t)(int)code;
    }
  }
  free(xs);
}

int wqo_w8a8_gemm_rows(const int8_t* Xq, const float* Sx, const int8_t* W,
                       const float* Sw, int M, int K, int N,
                       const int32_t* rows, int nrows,
                       int64_t* acc, double* y, double* abs_sum) {
  /* [QC] Dynamic Quantization: int8 multiply, int32 accumulate, then
   * Y = Sx * (Xint . Wint) * Sw. */
  (void)M;
  int overflow = 0;
  int64_t* absacc = (int64_t*)calloc((size_t)N, sizeof(int64_t));
  for (int r = 0; r < nrows; ++r) {
    int m = rows ? rows[r] : r;
    int64_t* a = acc + (size_t)r * N;
    for (int n = 0; n < N; ++n) { a[n] = 0; absacc[n] = 0; }
    for (int k = 0; k < K; ++k) {
      int64_t xq = Xq[(size_t)m * K + k];
      const int8_t* wrow = W + (size_t)k * N;
      for (int n = 0; n < N; ++n) {
        int64_t p = xq * (int64_t)wrow[n];
        a[n] += p;
        absacc[n] += p < 0 ? -p : p;
      }
    }
    for (int n = 0; n < N; ++n) {
      if (a[n] > 2147483647LL || a[n] < -2147483648LL) overflow = 1;
      double sxsw = (double)Sx[m] * (double)Sw[n];
      y[(size_t)r * N + n] = (double)Sx[m] * (double)a[n] * (double)Sw[n];
      abs_sum[(size_t)r * N + n] = sxsw * (double)absacc[n];
    }
  }
  free(absacc);
  return overflow;
}

/* ------------------------------------------------------------------------ */
/* LLM.int8() mixed-precision decomposition ([QC] LLM.int8(): the activation */
/* columns holding a value above the threshold, with the matching weight     */
/* rows, are multiplied in 16-bit floating point; the rest in int8; the two  */
/* results are added).                                                      */
/* ------------------------------------------------------------------------ */

void wqo_w8a8_outlier_columns(const uint16_t* X, int M, int K, float threshold, uint8_t* is_outlier) {
  for (int k = 0; k < K; ++k) {
    is_outlier[k] = 0;
    for (int m = 0; m < M; ++m)
      if (fabs(wqo_bf16_to_double(X[(size_t)m * K + k])) > (double)threshold) is_outlier[k] = 1;
  }
}

int wqo_w8a8_outlier_rows(const uint16_t* X, const uint8_t* is_outlier, const int8_t* Xq,
                          const float* Sx, const int8_t* W, const float* Sw, int M, int K, int N,
                          const int32_t* rows, int nrows, int64_t* acc, double* y, double* abs_sum) {
  /* int8 part: the regular columns (their codes; outlier columns have code 0),
   * exactly as wqo_w8a8_gemm_rows; 16-bit part: x[m,k] * Sw[n] * W[k,n] over
   * the outlier columns, with the activation as stored and the weight row
   * dequantized. */
  int overflow = wqo_w8a8_gemm_rows(Xq, Sx, W, Sw, M, K, N, rows, nrows, acc, y, abs_sum);
  for (int r = 0; r < nrows; ++r) {
    int m = rows ? rows[r] : r;
    for (int k = 0; k < K; ++k) {
      if (!is_outlier[k]) continue;
      double xv = wqo_bf16_to_double(X[(size_t)m * K + k]);
      for (int n = 0; n < N; ++n) {
        double t = xv * ((double)Sw[n] * (double)W[(size_t)k * N + n]);
        y[(size_t)r * N + n] += t;
        abs_sum[(size_t)r * N + n] += fabs(t);
      }
    }
  }
  return overflow;
}

