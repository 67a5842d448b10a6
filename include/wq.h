/*
 * wq.h -- C ABI of libwq.so: weight-only quantized GEMV / skinny GEMM with the
 * dequantization fused into the weight-tile load, and the W8A8 dynamic
 * quantization GEMM with an exact int32 product and a fused rescale epilogue.
 * Hand-written kernels for NVIDIA GB300 (sm_103a).
 *
 * Sources of the definitions (web pages, by title and section):
 *   [QC] "Quantization CUDA" (tom-jerr.github.io): Dynamic Quantization,
 *        优化 (fused rescale), Int8 Weight Only Quantization, Int4 Weight Only
 *        Quantization / Weight Store, Weight Only Quantization / 量化粒度,
 *        Marlin 格式.
 *   [GK] GPTQ CUDA kernel walkthrough (yelogs.com): CUDA核函數設計與實現 and
 *        C++封裝層實現 (vecquant3matmul(vec, mat, mul, scales, zeros)).
 *   [FD] "融合反量化与GEMM：LLM推理的CUDA内核优化实践" (zingnex.cn):
 *        核心优化思路 (dequantize inside the tile load, never write the
 *        dequantized weights back) and 量化策略：分组对称INT8.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every data pointer is a DEVICE pointer of the current CUDA device,
 *   owned by the caller; the library never allocates, frees or synchronizes.
 *   `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Calls are stream-ordered and asynchronous.
 * Layouts (row-major, no padding):
 *   x        [M, K]  activations;
 *   weights  K rows by N columns, N contiguous; packed formats pack
 *            consecutive k of ONE column into a 32-bit word:
 *              int8   : int8  [K, N];
 *              4-bit  : int32 [K/8, N], nibble j (bits 4j..4j+3) of word [r, n]
 *                       is the code of row 8r + j;
 *              3-bit  : int32 [3K/32, N]; the 32 codes of rows 32b..32b+31 of a
 *                       column form a 96-bit little-endian bit stream over word
 *                       rows 3b, 3b+1, 3b+2; code j occupies stream bits
 *                       [3j, 3j+3) (codes 10 and 21 straddle two words);
 *   scales   [K/group, N] (group-wise) or [N] (per column);
 *   qzeros   int32 [K/group, N/8], nibble j of word [g, c] = zero of column 8c+j;
 *   y        [M, N], overwritten (never accumulated into).
 * Alignment.  x, weights, scales, zeros, y (and W8A8 buffers) must be 16-byte
 *   aligned; N must be a multiple of 8 (16 for int8 weights).
 * Validation.  Every call validates all arguments before any CUDA call and
 *   returns an error with no side effect.  Launch failures are reported as
 *   WQ_ERR_CUDA (from cudaGetLastError right after the launch); errors that
 *   happen while the kernel runs surface at the caller's next synchronization.
 * Flags.  WQ_FLAG_PDL launches with programmatic dependent launch: the kernel
 *   may start while the preceding kernel on the stream is still running and
 *   prefetches its WEIGHTS, scales, zeros and g_idx before waiting for it; it
 *   waits before reading x and before writing anything.  Do not set it when the
 *   preceding kernel writes the weights.  0 = ordinary stream ordering.
 * Threads.  The library keeps no mutable global state: calls may be issued
 *   from several host threads and on several streams concurrently, provided
 *   their output and workspace buffers are distinct.
 */
#ifndef WQ_H
#define WQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define WQ_API __attribute__((visibility("default")))
#else
#define WQ_API
#endif

#define WQ_ABI_VERSION 1

typedef enum wq_status {
  WQ_OK = 0,
  WQ_ERR_NULL = 1,        /* a required pointer is NULL */
  WQ_ERR_SHAPE = 2,       /* M, K, N or group size out of range / not divisible */
  WQ_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
  WQ_ERR_UNSUPPORTED = 4, /* valid request this build does not implement (dtype, M) */
  WQ_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than the size query */
  WQ_ERR_CUDA = 6,        /* a CUDA runtime call or a launch failed */
  WQ_ERR_TIMEOUT = 7      /* reserved: a bounded device-side wait gave up */
} wq_status;

typedef enum wq_dtype { WQ_F16 = 1, WQ_BF16 = 2 } wq_dtype;

#define WQ_FLAG_PDL 1u

/* Human-readable name of a status code (static string, never NULL). */
WQ_API const char* wq_status_string(int status);

/* WQ_ABI_VERSION of the built library. */
WQ_API int wq_abi_version(void);

/* Value of the device-wide timeout flag of the current device: 1 if a bounded
 * device-side wait in any kernel of this library gave up since the flag was
 * last cleared (the outputs of that launch are then not valid), 0 otherwise,
 * -1 if the flag could not be read.  Synchronous (a device-to-host copy);
 * clear != 0 also resets it. */
WQ_API int wq_read_timeout_flag(int clear);

/*
 * wq8_gemv -- INT8 weight-only GEMV with group-wise fp32 scales.
 *   y[m,n] = sum_k x[m,k] * scales[k/group, n] * w[k,n]
 * [QC] Int8 Weight Only Quantization (Y = X.(Wint*Sw), fp32 accumulation);
 * [FD] 量化策略：分组对称INT8 (symmetric INT8, one scale per 128 along K).
 *   x      fp32 [M, K]      w      int8 [K, N]
 *   scales fp32 [K/group, N] y     fp32 [M, N]
 *   1 <= M <= 8; K >= 1, K % group == 0, group % 16 == 0; N % 16 == 0.
 */
WQ_API wq_status wq8_gemv(const float* x, const int8_t* w, const float* scales, float* y,
                          int M, int K, int N, int group_size, unsigned flags, void* stream);

/*
 * wq3_gemv -- 3-bit GEMV with per-column fp16 scale and stored fp16 zero.
 *   y[m,n] = sum_k x[m,k] * (scales[n] * q(k,n) - zeros[n])
 * where zeros[n] already holds scale * zero point.
 * [GK] CUDA核函數設計與實現 (res += (scale * q - zero) * vec[k]) and
 *      C++封裝層實現 (vecquant3matmul(vec, mat, mul, scales, zeros)).
 *   x      fp16 [M, K]      mat    int32 [3K/32, N]
 *   scales fp16 [N]         zeros  fp16 [N]        y  fp16 [M, N]
 *   1 <= M <= 8; K % 32 == 0; N % 8 == 0.  Accumulation is fp32.
 */
WQ_API wq_status wq3_gemv(const void* x, const int32_t* mat, const void* scales,
                          const void* zeros, void* y, int M, int K, int N,
                          unsigned flags, void* stream);

/*
 * wq4_gemm -- 4-bit group-wise weight-only GEMV / skinny GEMM.
 *   y[m,n] = sum_k x[m,k] * scales[g(k), n] * (q(k,n) - z(g(k), n))
 *   g(k) = g_idx[k] if g_idx != NULL (act-order), else k / group;
 *   z = the nibble of qzeros if qzeros != NULL, else 8 (symmetric).
 * [QC] 量化粒度 (x = S*(q - Z), group-wise), Marlin 格式 (eight INT4 per
 *      INT32, W = (Wint4 - Zero) * Scale), Int4 Weight Only Quantization.
 *   x      act_dtype [M, K]             qweight int32 [K/8, N]
 *   scales act_dtype [K/group, N]       qzeros  int32 [K/group, N/8] or NULL
 *   g_idx  int32 [K] with values in [0, K/group), or NULL
 *   y      act_dtype [M, N]
 *   act_dtype: WQ_F16 or WQ_BF16.  M >= 1; K % group == 0, group % 32 == 0;
 *   N % 8 == 0.  M <= 8 without g_idx runs on the warp-level tensor-core MMA
 *   when K % 64 == 0 and group % 64 == 0, else on CUDA cores; with g_idx it
 *   runs on CUDA cores (a scale gathered per code).  M > 8 runs on the
 *   tcgen05 tensor cores in chunks of up to 64 rows (padded to 16, 32 or 64)
 *   and needs group % 64 == 0 and g_idx == NULL; otherwise it returns
 *   WQ_ERR_UNSUPPORTED.
 *   workspace: none is needed; pass NULL and 0.
 */
WQ_API wq_status wq4_gemm(const void* x, const int32_t* qweight, const void* scales,
                          const int32_t* qzeros, const int32_t* g_idx, void* y,
                          int M, int K, int N, int group_size, int act_dtype,
                          void* workspace, size_t workspace_bytes,
                          unsigned flags, void* stream);

/*
 * wq4_actorder_prepare -- one-time preparation of act-order 4-bit weights for
 * wq4_gemm_sorted: sorts the rows of qweight by group, stable in k, so that
 * every group becomes a contiguous run of `group_size` rows.
 * [QC] Int4 Weight Only Quantization (group-wise); the act_order option of the
 *      GPTQ configuration (GPTQ算法解析, 4.1 内存-计算权衡).
 *   qweight        int32 [K/8, N]  input (device)
 *   g_idx          int32 [K]       input (device); every group must hold
 *                                  exactly group_size rows, else WQ_ERR_SHAPE
 *   qweight_sorted int32 [K/8, N]  output (device): sorted row i = row perm[i]
 *   perm           int32 [K]       output (device); g_idx[perm[i]] == i / group_size
 * Synchronous on `stream` (it reads g_idx back to the host); not for a hot path.
 */
WQ_API wq_status wq4_actorder_prepare(const int32_t* qweight, const int32_t* g_idx, int K, int N,
                                      int group_size, int32_t* qweight_sorted, int32_t* perm,
                                      void* stream);

/*
 * wq4_gemm_sorted -- the act-order GEMV on weights prepared by
 * wq4_actorder_prepare:
 *   y[m,n] = sum_i x[m, perm[i]] * scales[i/group, n] * (qs(i,n) - z(i/group, n))
 * which equals wq4_gemm with g_idx on the original weights (same scales and
 * qzeros: group ids do not change).  Each group is contiguous, so one scale
 * and zero apply per group instead of per code.
 *   1 <= M <= 8; K % group == 0, group % 32 == 0; N % 8 == 0; x (M*K values)
 *   must fit in shared memory next to the pipeline (M * K * 2 bytes <= about
 *   96 KB), else WQ_ERR_UNSUPPORTED.  Other arguments as in wq4_gemm.
 */
WQ_API wq_status wq4_gemm_sorted(const void* x, const int32_t* qweight_sorted, const void* scales,
                                 const int32_t* qzeros, const int32_t* perm, void* y, int M, int K,
                                 int N, int group_size, int act_dtype, unsigned flags, void* stream);

/*
 * wq4_repack_tiled -- one-time repack of 4-bit weights into the tile order of
 * the tensor-core GEMV (the offline weight reshuffle that "Quantization CUDA",
 * Marlin 格式 describes: a layout chosen so that the kernel's loads and the
 * MMA fragments line up; this layout is this library's own).
 *   Word (r, n) of the [K/8, N] matrix moves to
 *     ((r/8) * (N/32) + n/32) * 256 + ((r%8) % 2) * 128 + (4 ((n%32)/4) + (r%8)/2) * 4 + n%4
 *   so that each 64-value unit of k of each 32-column slab is one contiguous
 *   1 KB block and the blocks of one unit follow each other over the slabs.
 *   The codes inside each word are unchanged (nibble j = row 8r + j).
 *   qweight       int32 [K/8, N]  input (device), the wq4_gemm layout
 *   g_idx         int32 [K] or NULL (device): when given, the rows are first
 *                 sorted by group as wq4_actorder_prepare does (every group
 *                 must hold exactly group_size rows, else WQ_ERR_SHAPE), and
 *                 perm (int32 [K], device, output) receives the sort;
 *                 when NULL, perm is ignored and may be NULL
 *   qweight_tiled int32, (K/8) * N words, output (device)
 *   K % 64 == 0, N % 32 == 0, group_size % 64 == 0, K % group_size == 0.
 * Synchronous on `stream`; not for a hot path.
 */
WQ_API wq_status wq4_repack_tiled(const int32_t* qweight, const int32_t* g_idx, int K, int N,
                                  int group_size, int32_t* qweight_tiled, int32_t* perm, void* stream);

/*
 * wq4_gemm_tiled -- wq4_gemm (perm == NULL) or wq4_gemm_sorted (perm != NULL,
 * the perm written by wq4_repack_tiled) on weights repacked by
 * wq4_repack_tiled; same result, same scales and qzeros layouts.  Each
 * pipeline stage of a CTA's slab is one contiguous bulk copy.
 *   1 <= M <= 8; K % 64 == 0, N % 32 == 0, group_size = 64 * 2^j (64, 128,
 *   256, ...), K % group_size == 0; with perm, the CTA's K-slice of x is
 *   gathered into shared memory beside the pipeline; shapes whose shared
 *   memory does not fit return WQ_ERR_UNSUPPORTED.
 */
WQ_API wq_status wq4_gemm_tiled(const void* x, const int32_t* qweight_tiled, const void* scales,
                                const int32_t* qzeros, const int32_t* perm, void* y, int M, int K,
                                int N, int group_size, int act_dtype, unsigned flags, void* stream);

/*
 * wq8_dequant / wq3_dequant / wq4_dequant -- standalone dequantization: the
 * packed weights of wq8_gemv / wq3_gemv / wq4_gemm expanded into a dense
 * row-major [K, N] matrix in device memory.  This is the separate-kernel path
 * that fusion removes ("融合反量化与GEMM：LLM推理的CUDA内核优化实践",
 * 核心优化思路 and CUDA内核架构: dequantize into a DRAM buffer, then a separate
 * GEMM), kept as a baseline and for callers that want dense weights (for
 * example to run a large-M product through a dense GEMM library).
 *   wq8_dequant: w_out fp32 [K, N], w_out[k,n] = fp32(scales[k/g, n] * w[k,n])
 *                (one rounding of the exact product).  Same shapes, group and
 *                alignment rules as wq8_gemv.
 *   wq3_dequant: w_out fp16 [K, N], w_out[k,n] = fp16(fp32 fma(s[n], q(k,n),
 *                -zeros[n])): rounded once to fp32 and then to fp16, which is
 *                the exact value rounded once whenever s[n]*q - zeros[n] fits
 *                in 24 bits (always, for scales and zeros within a factor 2^10
 *                of each other).  Same shape rules as wq3_gemv.
 *   wq4_dequant: w_out [K, N] in act_dtype (fp16 or bf16),
 *                w_out[k,n] = act(s[g(k), n] * (q(k,n) - z[g(k), n])), g(k) =
 *                g_idx[k] (values outside [0, K/group) are clamped) or k/group,
 *                z = 8 when qzeros is NULL: the product is exact in fp32 and
 *                rounded once.  Same shape and alignment rules as wq4_gemm.
 * All pointers are device pointers owned by the caller; w_out must not alias
 * the inputs and must be 16-byte aligned.  Asynchronous on `stream`; flags may
 * hold WQ_FLAG_PDL.  Errors: WQ_ERR_NULL, WQ_ERR_SHAPE, WQ_ERR_ALIGN,
 * WQ_ERR_UNSUPPORTED (act_dtype), WQ_ERR_CUDA (launch failure); nothing runs
 * on an argument error.
 */
WQ_API wq_status wq8_dequant(const int8_t* w, const float* scales, float* w_out, int K, int N,
                             int group_size, unsigned flags, void* stream);
WQ_API wq_status wq3_dequant(const int32_t* mat, const void* scales, const void* zeros,
                             void* w_out, int K, int N, unsigned flags, void* stream);
WQ_API wq_status wq4_dequant(const int32_t* qweight, const void* scales, const int32_t* qzeros,
                             const int32_t* g_idx, void* w_out, int K, int N, int group_size,
                             int act_dtype, unsigned flags, void* stream);

/*
 * w8a8_gemm -- W8A8 dynamic-quantization GEMM.
 *   Sx[m]    = fp32(max_k |X[m,k]| / 127)              (fp32 division)
 *   Xq[m,k]  = clamp(rint(fp32(X[m,k] / Sx[m])), -127, 127)   (ties to even;
 *              an all-zero row has Sx = 0 and Xq = 0)
 *   acc[m,n] = sum_k Xq[m,k] * W[k,n]                  (exact int32)
 *   Y[m,n]   = bf16(Sx[m] * acc[m,n] * Sw[n])          (the int32 product is
 *              never stored unless acc_out is given)
 * [QC] Dynamic Quantization (Y = Sx*(Xint.Wint)*Sw, int8 multiply, int32
 *      accumulate, float rescale), 优化 (multiply fused into the matmul so the
 *      int32 result is not materialized), 量化粒度 (per-token, per-channel).
 *   X    bf16 [M, K]     W  int8 [K, N]     Sw  fp32 [N]     Y  bf16 [M, N]
 *   Xq_out int8 [M, K] or NULL; Sx_out fp32 [M] or NULL;
 *   acc_out int32 [M, N] or NULL (debug: writes the exact product);
 *   workspace >= w8a8_gemm_workspace_bytes(M, K, N) bytes, 256-byte aligned.
 *   M >= 1; K % 64 == 0, K <= 65536; N % 16 == 0.
 */
WQ_API wq_status w8a8_gemm(const void* X, const int8_t* W, const float* Sw, void* Y,
                           int M, int K, int N, int8_t* Xq_out, float* Sx_out,
                           int32_t* acc_out, void* workspace, size_t workspace_bytes,
                           unsigned flags, void* stream);

/*
 * w8a8_gemm_smooth -- w8a8_gemm with Smoothquant's activation side
 * ([QC] Smoothquant: Y = (X diag(s)^-1) . (diag(s) W), which moves the
 * quantization difficulty of outlier activation channels onto the weights):
 *   X'[m,k] = fp32(X[m,k] / smooth[k])     (one correctly rounded division)
 * and then everything w8a8_gemm does, on X' instead of X (Sx, Xq_out and
 * Sx_out describe X').  The caller supplies W as the int8 codes of diag(s) W
 * with their per-column Sw, prepared offline.
 *   smooth fp32 [K], device, 16-byte aligned; every entry finite and > 0 (not
 *   checked: it is device data; other values give meaningless codes).
 *   Everything else as in w8a8_gemm (same errors; smooth NULL is WQ_ERR_NULL).
 */
WQ_API wq_status w8a8_gemm_smooth(const void* X, const float* smooth, const int8_t* W,
                                  const float* Sw, void* Y, int M, int K, int N,
                                  int8_t* Xq_out, float* Sx_out, int32_t* acc_out,
                                  void* workspace, size_t workspace_bytes, unsigned flags,
                                  void* stream);

/*
 * w8a8_gemm_outlier -- W8A8 with LLM.int8()'s mixed-precision decomposition
 * ([QC] LLM.int8(): the activation columns holding a value above a threshold,
 * with the matching weight rows, stay in 16-bit floating point; the rest goes
 * through int8; the two results are added):
 *   O        = { k : |X[m,k]| > threshold for some m }   (strictly greater)
 *   Sx, Xq   = the row quantization of w8a8_gemm applied to X with the
 *              columns in O set to zero (the regular part)
 *   acc[m,n] = sum_k Xq[m,k] * W[k,n]                     (exact int32)
 *   Y[m,n]   = bf16( (Sx[m]*acc[m,n])*Sw[n]
 *                    + sum_{k in O} X[m,k] * (Sw[n]*W[k,n]) )  (fp32)
 * The 16-bit part uses the activations as stored (bf16) and the weight rows
 * dequantized from their int8 codes; it is added in fp32 before the single
 * bf16 rounding of Y.  threshold: any float (the pages use 6.0; a negative
 * value sends every column to the 16-bit part, +inf none).
 *   n_outliers_out: device int32 or NULL, receives |O|.
 *   workspace >= w8a8_gemm_outlier_workspace_bytes(M, K, N) bytes, 256-byte
 *   aligned.  Other arguments, shapes and errors as in w8a8_gemm.
 */
WQ_API wq_status w8a8_gemm_outlier(const void* X, const int8_t* W, const float* Sw, void* Y,
                                   int M, int K, int N, float threshold, int8_t* Xq_out,
                                   float* Sx_out, int32_t* acc_out, int32_t* n_outliers_out,
                                   void* workspace, size_t workspace_bytes, unsigned flags,
                                   void* stream);

/* Bytes of device workspace w8a8_gemm_outlier needs for this shape (0 on bad
 * shape): the workspace of w8a8_gemm, the column flags and the list of outlier
 * columns (4 K bytes each), and room for the gathered bf16 activations of up
 * to K outlier columns (2 K M bytes). */
WQ_API size_t w8a8_gemm_outlier_workspace_bytes(int M, int K, int N);

/* Bytes of device workspace w8a8_gemm needs for this shape (0 on bad shape). */
WQ_API size_t w8a8_gemm_workspace_bytes(int M, int K, int N);

/*
 * w8a8_gemm_noalloc -- w8a8_gemm without a caller workspace.  The pages have
 * no counterpart: this is library plumbing, not part of the method.
 *
 * Who it is for: callers that cannot allocate device memory for the
 *   workspace -- code whose device memory is owned by someone else (a host
 *   framework or server that reserves all of it up front), code with a fixed
 *   memory budget, and code that must not pay for cudaMalloc / cudaFree, which
 *   can block and (cudaFree) synchronize the whole device.  This entry point
 *   allocates nothing: it runs w8a8_gemm on a scratch array built into the
 *   library, one copy per device, of w8a8_gemm_noalloc_max_scratch_bytes()
 *   bytes (8 MiB).
 * Arguments, layouts, results and checks: as w8a8_gemm, without `workspace`.
 * Size limit: the shape's w8a8_gemm_workspace_bytes(M, K, N) =
 *   align256(2*M*K) + align256(4*M) must not exceed the built-in size (for
 *   example M <= 511 at K = 8192, M <= 1023 at K = 4096);
 *   a larger shape returns WQ_ERR_WORKSPACE before anything runs -- use
 *   w8a8_gemm with a workspace of your own for it.
 * First call on each device: looks up the device address of the built-in
 *   scratch (the CUDA runtime may load the library's device code then) and
 *   caches it.  This set-up is done with the caller's current device, once
 *   per device; make the first call on each device before any stream
 *   capture begins.  A failed look-up returns WQ_ERR_CUDA.
 * Zero state: nothing needs to start at zero; every call writes each scratch
 *   byte it later reads.
 * Concurrency: all calls on one device share the one scratch array.  Calls
 *   whose executions can overlap -- on different streams without an ordering
 *   between them, from any thread -- race on it and may return wrong
 *   results.  Calls issued on one stream (or otherwise ordered) are safe,
 *   also back to back with WQ_FLAG_PDL: the call's first kernel waits for the
 *   preceding grid on the stream to complete before it writes the scratch.
 */
WQ_API wq_status w8a8_gemm_noalloc(const void* X, const int8_t* W, const float* Sw, void* Y,
                                   int M, int K, int N, int8_t* Xq_out, float* Sx_out,
                                   int32_t* acc_out, unsigned flags, void* stream);

/* Bytes of the scratch array w8a8_gemm_noalloc uses (the size limit above). */
WQ_API size_t w8a8_gemm_noalloc_max_scratch_bytes(void);

#ifdef __cplusplus
}
#endif
#endif /* WQ_H */
