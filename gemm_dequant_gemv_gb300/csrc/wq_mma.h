// wq_mma.h -- host-side interface of the tensor-core paths (tcgen05): the
// 4-bit weight-only GEMM for M >= 16 and the W8A8 dynamic-quantization GEMM.
// Internal to libwq.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace wq {

cudaError_t launch_wq4_mma(const void* x, const int32_t* qweight, const void* scales, const int32_t* qzeros,
                           void* y, int M, int K, int N, int group, int act_bf16, unsigned flags,
                           cudaStream_t stream);

size_t w8a8_workspace_bytes(int M, int K, int N);

// smooth: Smoothquant's per-channel divisor of the activations (fp32 [K]), or null.
// outlier_threshold: LLM.int8()'s threshold (host value), or null; then the
// workspace holds w8a8_outlier_workspace_bytes and n_outliers_out (device,
// optional) receives the number of outlier columns.
cudaError_t launch_w8a8(const void* X, const int8_t* W, const float* Sw, void* Y, int M, int K, int N,
                        int8_t* Xq_out, float* Sx_out, int32_t* acc_out, void* workspace, unsigned flags,
                        cudaStream_t stream, const float* smooth = nullptr,
                        const float* outlier_threshold = nullptr, int32_t* n_outliers_out = nullptr);
size_t w8a8_outlier_workspace_bytes(int M, int K, int N);

// Act-order preparation (host-driven, synchronous on `stream`): 0 = ok,
// 1 = g_idx is not a grouping with exactly `group` rows per group, 2 = CUDA error.
// The tensor-core GEMV's tiled layout (host-driven, synchronous on `stream`):
// rows sorted by group first when g_idx != null (perm written then); same
// return codes as actorder_prepare.
int repack_tiled(const int32_t* qweight, const int32_t* g_idx, int K, int N, int group, int32_t* qweight_tiled,
                 int32_t* perm, cudaStream_t stream);

int actorder_prepare(const int32_t* qweight, const int32_t* g_idx, int K, int N, int group, int32_t* qweight_sorted,
                     int32_t* perm, cudaStream_t stream);

}  // namespace wq
