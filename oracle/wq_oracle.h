/*
 * wq_oracle.h -- plain CPU oracle for weight-only quantized GEMV/GEMM and the
 * W8A8 dynamic-quantization GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this code; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no source with the CUDA path.
 *
 * Every routine is single-threaded, accumulates in double (or int64 for the
 * integer product) and decodes the packed weight formats with its own bit
 * arithmetic.  Outputs are the exact-arithmetic value of the definition before
 * any rounding to the output dtype, plus the per-output magnitude sum
 *   abs[m,n] = sum_k |x[m,k] * w(k,n)|
 * that the numerical tolerance is stated against.
 *
 * Layout conventions (shared with the product, restated here so the oracle can
 * be read on its own):
 *   - activations x: row-major [M, K];
 *   - weights: row-major over K rows and N columns, N contiguous; packed
 *     formats pack consecutive k of one column n into one 32-bit word;
 *   - outputs: row-major [M, ncols] over the requested columns.
 *
 * Parity pins: every function here is pinned by the CPU tests (hand-worked
 * words, closed forms, library reductions and invariants); none is unpinned.
 */
#ifndef WQ_ORACLE_H
#define WQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- scalar formats (IEEE 754 binary16, bfloat16) ---------------------- */
double   wqo_f16_to_double(uint16_t h);
double   wqo_bf16_to_double(uint16_t b);
uint16_t wqo_double_to_f16(double v);   /* round to nearest, ties to even */
uint16_t wqo_double_to_bf16(double v);  /* round to nearest, ties to even */
float    wqo_double_to_f32(double v);   /* round to nearest, ties to even */

/* ---- code extraction from the packed formats ---------------------------- */
/* 3-bit: 32 codes of k = 32b..32b+31 form a 96-bit little-endian bit stream
 * over word rows 3b, 3b+1, 3b+2 of column n; code j sits at bits [3j, 3j+3). */
int wqo_code3(const int32_t* mat, int N, int k, int n);
/* 4-bit: nibble j (bits [4j, 4j+4)) of word row k/8 of column n is code k. */
int wqo_code4(const int32_t* qweight, int N, int k, int n);
/* 4-bit zeros: nibble j of word [g, c] is the zero point of column 8c + j. */
int wqo_zero4(const int32_t* qzeros, int N, int g, int n);

/* Unpack whole matrices (codes as uint8, row-major [K, N] / [G, N]). */
void wqo_unpack3(const int32_t* mat, int K, int N, uint8_t* codes);
void wqo_unpack4(const int32_t* qweight, int K, int N, uint8_t* codes);
void wqo_unpack_zeros4(const int32_t* qzeros, int G, int N, uint8_t* zeros);

/* ---- the products --------------------------------------------------------
 * cols: the output columns to compute (ncols of them), or NULL for all N (then
 * ncols must equal N).  y and abs_sum are [M, ncols] row-major doubles. */

/* 8-bit symmetric, group-wise fp32 scales [K/group, N]:
 *   w(k,n) = scales[k/group, n] * q[k,n]. */
void wqo_wq8_gemv(const float* x, const int8_t* w, const float* scales,
                  int M, int K, int N, int group,
                  const int32_t* cols, int ncols, double* y, double* abs_sum);

/* 3-bit, per-column fp16 scale and fp16 stored zero (already scale * z):
 *   w(k,n) = scales[n] * q[k,n] - zeros[n]. x is fp16 [M, K]. */
void wqo_wq3_gemv(const uint16_t* x, const int32_t* mat, const uint16_t* scales,
                  const uint16_t* zeros, int M, int K, int N,
                  const int32_t* cols, int ncols, double* y, double* abs_sum);

/* ---- dequantization (the unfused baseline: dense weights in memory) -------
 * The exact value of every weight, w(k,n) by the formulas of the products
 * below, as a dense row-major [K, N] double matrix. */
void wqo_wq8_dequant(const int8_t* w, const float* scales, int K, int N, int group, double* out);
void wqo_wq3_dequant(const int32_t* mat, const uint16_t* scales, const uint16_t* zeros,
                     int K, int N, double* out);
void wqo_wq4_dequant(int act_bf16, const int32_t* qweight, const uint16_t* scales,
                     const int32_t* qzeros, const int32_t* g_idx, int K, int N, int group,
                     double* out);

/* 4-bit, group-wise scales [K/group, N] in the activation dtype, 4-bit zeros
 * [K/group, N/8] (NULL: every zero is 8), optional act-order g_idx [K]
 * (NULL: group of row k is k/group):
 *   w(k,n) = scales[g(k), n] * (q[k,n] - z[g(k), n]).
 * act_bf16 = 0: x and scales are fp16; 1: bf16. */
void wqo_wq4_gemm(const uint16_t* x, int act_bf16, const int32_t* qweight,
                  const uint16_t* scales, const int32_t* qzeros,
                  const int32_t* g_idx, int M, int K, int N, int group,
                  const int32_t* cols, int ncols, double* y, double* abs_sum);

/* W8A8 step 1, per-row dynamic quantization of bf16 X [M, K]:
 *   Sx[m] = fp32(max_k |X[m,k]| / 127)   (fp32 division, correctly rounded)
 *   Xq    = clamp(round_half_even(fp32(X / Sx[m])), -127, 127); Sx = 0 => 0. */
void wqo_w8a8_quant_rows(const uint16_t* X, int M, int K, int8_t* Xq, float* Sx);

/* W8A8 steps 2 and 3 for the listed rows (nrows of them; NULL = all M, then
 * nrows == M) and all N columns:
 *   acc[r, n] = sum_k Xq[m,k] * W[k,n]            (int64, exact)
 *   y[r, n]   = Sx[m] * acc[r, n] * Sw[n]          (double, before rounding)
 *   abs_sum   = sum_k |Sx[m] Xq[m,k] * Sw[n] W[k,n]|
 * Returns 0 if every acc fits int32, else 1. */
/* Smoothquant's run-time half: X'[m,k] = fp32(X[m,k] / smooth[k]), then the
 * per-row quantization of wqo_w8a8_quant_rows applied to X' (the weights are
 * the caller's int8 codes of diag(s) W, prepared offline). */
void wqo_w8a8_quant_rows_smooth(const uint16_t* X, const float* smooth, int M, int K, int8_t* Xq,
                                float* Sx);

int wqo_w8a8_gemm_rows(const int8_t* Xq, const float* Sx, const int8_t* W,
                       const float* Sw, int M, int K, int N,
                       const int32_t* rows, int nrows,
                       int64_t* acc, double* y, double* abs_sum);

/* LLM.int8() decomposition: is_outlier[k] = 1 when some |X[m,k]| > threshold
 * (strictly greater).  wqo_w8a8_outlier_rows takes Xq / Sx of X with the
 * outlier columns set to zero (the regular part) and returns
 *   y[m,n] = Sx[m] * sum_k Xq[m,k] W[k,n] * Sw[n]
 *          + sum_{k outlier} X[m,k] * (Sw[n] * W[k,n])
 * with acc the int8 part's exact sum and abs_sum the magnitude sum of both
 * parts; the return value is 1 if an int8 sum leaves int32. */
void wqo_w8a8_outlier_columns(const uint16_t* X, int M, int K, float threshold, uint8_t* is_outlier);
int wqo_w8a8_outlier_rows(const uint16_t* X, const uint8_t* is_outlier, const int8_t* Xq,
                          const float* Sx, const int8_t* W, const float* Sw, int M, int K, int N,
                          const int32_t* rows, int nrows, int64_t* acc, double* y, double* abs_sum);

#ifdef __cplusplus
}
#endif
#endif /* WQ_ORACLE_H */
