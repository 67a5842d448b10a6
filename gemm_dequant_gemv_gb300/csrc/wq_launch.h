// wq_launch.h -- host-side interface between the C ABI (wq_api.cu) and the
// kernel files.  Internal to libwq.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace wq {

struct GemvArgs;

// How a GEMV-family kernel is launched: T column tiles (grid.y) x S K-slices
// (grid.x, one thread-block cluster of S CTAs per tile), MT = rows of x the
// kernel instance handles (1, 2, 4 or 8).
struct LaunchPlan {
  int T, S, MT;
  unsigned flags;
  cudaStream_t stream;
};

// Generic launcher: cluster dims (S,1,1) when S > 1, programmatic dependent
// launch when flags has WQ_FLAG_PDL.  `kern` takes nmaps CUtensorMaps
// (__grid_constant__) followed by the GemvArgs.
cudaError_t launch_gemv_kernel(const void* kern, const LaunchPlan& p, size_t smem_bytes,
                               const CUtensorMap* const* maps, int nmaps, const GemvArgs& a);

size_t wq8_gemv_smem_bytes(int MT, int ng_max, int S);
size_t wq3_gemv_smem_bytes(int MT, int S);
size_t wq4_gemv_smem_bytes(int MT, int ng_max, bool act_order, int G, int S, size_t xfull_bytes = 0);

// Values of k one pipeline stage covers (the x box width of each kernel).
int wq8_stage_k();
int wq3_stage_k();
int wq4_stage_k();

cudaError_t launch_wq8_gemv(const LaunchPlan& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                            const GemvArgs& a);
cudaError_t launch_wq3_gemv(const LaunchPlan& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                            const GemvArgs& a);
// gmap != nullptr selects the act-order kernel (g_idx staged per stage);
// sorted selects the kernel for group-sorted rows, with xmap mapping perm.
cudaError_t launch_wq4_gemv(const LaunchPlan& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                            const CUtensorMap* gmap, const GemvArgs& a, int act_bf16, bool has_z,
                            bool sorted = false);

// 4-bit GEMV on the warp-level tensor-core MMA (contiguous groups, or rows
// sorted by group when perm): needs K % wq4m_unit_k() == 0 and a group size
// that is a multiple of it; the weight map uses 32 x 32 boxes, 128-byte swizzle.
int wq4m_unit_k();
int wq4m_stage_k();
size_t wq4m_gemv_smem_bytes(int MT, int ng_max, int S, bool perm, int K);
cudaError_t launch_wq4m_gemv(const LaunchPlan& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                             const GemvArgs& a, int act_bf16, bool has_z, bool perm);

// 4-bit GEMV on the warp-level tensor-core MMA with variable-width column
// tiles (wq_gemv4t.cu); the tile shape and K-split are planned per call.
struct Plan4T {
  int nslab, S, T, NS, MT;
};
int wq4t_unit_k();
// qweight: GPTQ layout [K/8, N] (wtiled == nullptr), or wtiled: the layout of
// wq4_repack_tiled; perm != nullptr: rows sorted by act-order group.
// Returns cudaErrorNotSupported for shapes this kernel does not take (M > 8,
// K % 64, a group that is not 64 times a power of two, shared memory).
cudaError_t launch_wq4t(const void* x, const int32_t* qweight, const uint8_t* wtiled, const void* scales,
                        const int32_t* qzeros, const int32_t* perm, void* y, int M, int K, int N, int group,
                        int act_bf16, unsigned flags, cudaStream_t stream);

// 3-bit GEMV with per-column scale and stored zero on the warp-level
// tensor-core MMA (wq_gemv3t.cu), planned per call.  cudaErrorNotSupported
// for shapes it does not take (M > 8, K % 32, N % 8, shared memory).
cudaError_t launch_wq3t(const void* x, const int32_t* mat, const void* scales, const void* zeros, void* y, int M,
                        int K, int N, unsigned flags, cudaStream_t stream);

// Device queries and tensor-map encoding (wq_api.cu).
int device_sm_count();
// Clusters of S CTAs of `threads` threads and `smem` bytes of dynamic shared
// memory each that the device runs at once for kernel `kern` (S == 1: CTAs);
// cached per device and configuration, 0 for a shape the device cannot run.
int cluster_capacity(const void* kern, int S, int threads, size_t smem);
int device_max_smem();
bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swizzle);

// Standalone dequantization to a dense [K, N] matrix (wq_dequant.cu).
cudaError_t launch_wq8_dequant(const int8_t* w, const float* scales, float* out, int K, int N, int group,
                               unsigned flags, cudaStream_t stream);
cudaError_t launch_wq3_dequant(const int32_t* mat, const void* scales, const void* zeros, void* out, int K, int N,
                               unsigned flags, cudaStream_t stream);
cudaError_t launch_wq4_dequant(const int32_t* qweight, const void* scales, const int32_t* qzeros,
                               const int32_t* g_idx, void* out, int K, int N, int group, int act_bf16,
                               unsigned flags, cudaStream_t stream);

}  // namespace wq
