// wq_api.cu -- the C ABI of libwq.so: argument validation, tensor-map
// encoding, launch planning and dispatch to the kernels.  See include/wq.h for
// the contract of every entry point.
#include <cudaTypedefs.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/wq.h"
#include "wq_gemv_common.cuh"
#include "wq_launch.h"
#include "wq_mma.h"

namespace wq {

__device__ unsigned int g_timeout_flag = 0;

namespace {

constexpr int kMaxDim = 1 << 24;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled through the runtime's driver entry point, so that the
// library has no link-time dependency on libcuda.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

// 2D row-major tensor [outer, inner] of `dt` elements, box [box_outer, box_inner],
// no swizzle, out-of-bounds elements read as zero.
bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swizzle) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int device_max_smem() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  return n;
}

// Clusters of S CTAs (threads, smem each) the device runs at once, per
// kernel instance and configuration; looked up once and cached (the only
// process-wide state besides the tensor-map encoder, guarded by a mutex).
int cluster_capacity(const void* kern, int S, int threads, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, int, size_t>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const auto key = std::make_tuple(dev, kern, S, threads, smem);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return 0;
  if (S == 1) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess) return 0;
    n = per_sm * device_sm_count();
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      cudaGetLastError();  // an unsupported cluster shape: report no capacity
      n = 0;
    }
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = n;
  return n;
}

cudaError_t launch_gemv_kernel(const void* kern, const LaunchPlan& p, size_t smem_bytes,
                               const CUtensorMap* const* maps, int nmaps, const GemvArgs& a) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.S, p.T, 1);
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = p.stream;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (p.S > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = p.S;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  if (p.flags & WQ_FLAG_PDL) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  void* args[4];
  for (int i = 0; i < nmaps; ++i) args[i] = const_cast<CUtensorMap*>(maps[i]);
  args[nmaps] = const_cast<GemvArgs*>(&a);
  return cudaLaunchKernelExC(&cfg, kern, args);
}

namespace {

// K-slices per column tile: about two CTAs per SM (two fit in shared memory,
// so the next kernel's prologue can overlap this one's tail), at most 8 (a
// portable cluster) and at most one slice per work unit.
int plan_splits(int tiles, int units) {
  const int sms = std::max(1, device_sm_count());
  int s = (2 * sms) / tiles;
  s = std::max(1, std::min(s, 8));
  return std::min(s, std::max(units, 1));
}

// Activation map: [rows, K] elements of `dt`, box = one stage's k by MT rows.
bool encode_x_map(CUtensorMap* map, CUtensorMapDataType dt, const void* x, int K, int M, int esize, int stage_k,
                  int MT) {
  return encode_tensor_map_2d(map, dt, x, K, M, size_t(K) * esize, stage_k, MT, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Most scale groups any one of the S K-slices touches.
int max_groups_per_slice(int units, int S, int unit_k, int group) {
  int mx = 1;
  for (int s = 0; s < S; ++s) {
    const int u0 = static_cast<int>((static_cast<long long>(s) * units) / S);
    const int u1 = static_cast<int>((static_cast<long long>(s + 1) * units) / S);
    if (u1 > u0) mx = std::max(mx, (unit_k * u1 - 1) / group - (unit_k * u0) / group + 1);
  }
  return mx;
}

int round_mt(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

wq_status from_cuda(cudaError_t e) {
  if (e == cudaErrorNotSupported) return WQ_ERR_UNSUPPORTED;
  return e == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

// The tensor-core 4-bit GEMV (2 <= M <= 8, group a multiple of its 64-value unit;
// K % group == 0 was checked by the caller).  perm != nullptr: rows sorted by group.
// For M = 1 the CUDA-core kernels are as fast or faster on GB300 (measured:
// 44 vs 46 us at 8192 x 28672, 10.9 vs 11.6 us for the sorted 4096 x 11008),
// while from M = 2 on the MMA path costs the same as M = 1 and the CUDA-core
// one grows with M.
wq_status wq4m_launch(const void* x, const int32_t* qweight, const void* scales, const int32_t* qzeros,
                      const int32_t* perm, void* y, int M, int K, int N, int group_size, int act_bf16,
                      unsigned flags, cudaStream_t stream) {
  const int T = (N + 127) / 128, units = K / wq4m_unit_k();
  LaunchPlan p{T, plan_splits(T, units), round_mt(M), flags, stream};
  GemvArgs a{x, y, scales, qzeros, nullptr, M, K, N, group_size, 0};
  a.ng_max = max_groups_per_slice(units, p.S, wq4m_unit_k(), group_size);
  if (wq4m_gemv_smem_bytes(p.MT, a.ng_max, p.S, perm != nullptr, K) > static_cast<size_t>(device_max_smem()))
    return WQ_ERR_UNSUPPORTED;
  CUtensorMap wmap, xmap;
  if (!encode_tensor_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, qweight, N, K / 8, size_t(N) * 4, 32, 32,
                            CU_TENSOR_MAP_SWIZZLE_128B))
    return WQ_ERR_CUDA;
  if (perm ? !encode_x_map(&xmap, CU_TENSOR_MAP_DATA_TYPE_INT32, perm, K, 1, 4, wq4m_stage_k(), 1)
           : !encode_x_map(&xmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, x, K, M, 2, wq4m_stage_k(), p.MT))
    return WQ_ERR_CUDA;
  return from_cuda(launch_wq4m_gemv(p, wmap, xmap, a, act_bf16, qzeros != nullptr, perm != nullptr));
}

}  // namespace
}  // namespace wq

using namespace wq;

extern "C" {

WQ_API const char* wq_status_string(int status) {
  switch (status) {
    case WQ_OK: return "ok";
    case WQ_ERR_NULL: return "a required pointer is NULL";
    case WQ_ERR_SHAPE: return "a shape or group-size argument is out of range or not divisible";
    case WQ_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case WQ_ERR_UNSUPPORTED: return "request not supported by this build";
    case WQ_ERR_WORKSPACE: return "workspace missing or too small";
    case WQ_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case WQ_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    default: return "unknown status";
  }
}

WQ_API int wq_abi_version(void) { return WQ_ABI_VERSION; }

WQ_API int wq_read_timeout_flag(int clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_timeout_flag, sizeof v) != cudaSuccess) return -1;
  if (clear && v) {
    const unsigned int z = 0;
    if (cudaMemcpyToSymbol(g_timeout_flag, &z, sizeof z) != cudaSuccess) return -1;
  }
  return static_cast<int>(v);
}

WQ_API wq_status wq8_gemv(const float* x, const int8_t* w, const float* scales, float* y, int M, int K, int N,
                          int group_size, unsigned flags, void* stream) {
  if (!x || !w || !scales || !y) return WQ_ERR_NULL;
  if (M < 1 || M > 8 || K < 1 || N < 1 || K > kMaxDim || N > kMaxDim) return WQ_ERR_SHAPE;
  if (group_size < 16 || group_size % 16 != 0 || K % group_size != 0 || N % 16 != 0) return WQ_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(scales) || !aligned16(y)) return WQ_ERR_ALIGN;

  const int T = (N + 127) / 128, units = K / 16;
  LaunchPlan p{T, plan_splits(T, units), round_mt(M), flags, static_cast<cudaStream_t>(stream)};
  GemvArgs a{x, y, scales, nullptr, nullptr, M, K, N, group_size, 0};
  a.ng_max = max_groups_per_slice(units, p.S, 16, group_size);
  if (wq8_gemv_smem_bytes(p.MT, a.ng_max, p.S) > static_cast<size_t>(device_max_smem())) return WQ_ERR_UNSUPPORTED;
  CUtensorMap wmap, xmap;
  if (!encode_tensor_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, N, K, N, 128, wq8_stage_k(),
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_x_map(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, x, K, M, 4, wq8_stage_k(), p.MT))
    return WQ_ERR_CUDA;
  return from_cuda(launch_wq8_gemv(p, wmap, xmap, a));
}

WQ_API wq_status wq3_gemv(const void* x, const int32_t* mat, const void* scales, const void* zeros, void* y, int M,
                          int K, int N, unsigned flags, void* stream) {
  if (!x || !mat || !scales || !zeros || !y) return WQ_ERR_NULL;
  if (M < 1 || M > 8 || K < 32 || N < 1 || K > kMaxDim || N > kMaxDim) return WQ_ERR_SHAPE;
  if (K % 32 != 0 || N % 8 != 0) return WQ_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(mat) || !aligned16(scales) || !aligned16(zeros) || !aligned16(y))
    return WQ_ERR_ALIGN;

  // M >= 3: the tensor-core kernel (its MMAs cost the same for any M <= 8),
  // where its pair-ordered x fits in shared memory; M <= 2 and the rest: the
  // CUDA-core kernel (faster there: 5.0 against 5.4 us at M = 1, chained)
  if (M >= 3) {
    const cudaError_t e = launch_wq3t(x, mat, scales, zeros, y, M, K, N, flags, static_cast<cudaStream_t>(stream));
    if (e != cudaErrorNotSupported) return from_cuda(e);
  }
  const int T = (N + 127) / 128, units = K / 32;
  LaunchPlan p{T, plan_splits(T, units), round_mt(M), flags, static_cast<cudaStream_t>(stream)};
  GemvArgs a{x, y, scales, zeros, nullptr, M, K, N, 0, 0};
  if (wq3_gemv_smem_bytes(p.MT, p.S) > static_cast<size_t>(device_max_smem())) return WQ_ERR_UNSUPPORTED;
  CUtensorMap wmap, xmap;
  if (!encode_tensor_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, mat, N, 3 * (K / 32), size_t(N) * 4, 128, 24,
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_x_map(&xmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, x, K, M, 2, wq3_stage_k(), p.MT))
    return WQ_ERR_CUDA;
  return from_cuda(launch_wq3_gemv(p, wmap, xmap, a));
}

WQ_API wq_status wq4_gemm(const void* x, const int32_t* qweight, const void* scales, const int32_t* qzeros,
                          const int32_t* g_idx, void* y, int M, int K, int N, int group_size, int act_dtype,
                          void* workspace, size_t workspace_bytes, unsigned flags, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (!x || !qweight || !scales || !y) return WQ_ERR_NULL;
  if (M < 1 || K < 32 || N < 1 || K > kMaxDim || N > kMaxDim) return WQ_ERR_SHAPE;
  if (group_size < 32 || group_size % 32 != 0 || K % group_size != 0 || N % 8 != 0) return WQ_ERR_SHAPE;
  if (act_dtype != WQ_F16 && act_dtype != WQ_BF16) return WQ_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(qweight) || !aligned16(scales) || !aligned16(y) ||
      (qzeros && !aligned16(qzeros)) || (g_idx && !aligned16(g_idx)))
    return WQ_ERR_ALIGN;
  const int act_bf16 = act_dtype == WQ_BF16;

  if (M > 8) {
    if (g_idx) return WQ_ERR_UNSUPPORTED;
    // up to 32 rows: the warp-level MMA kernel with two or four n-tiles (the
    // conversion of each code serves every row, and it measured about twice
    // as fast as the tcgen05 kernel there); beyond, the tcgen05 kernel
    if (M <= 32 && K % wq4t_unit_k() == 0 && group_size % wq4t_unit_k() == 0) {
      const cudaError_t e = launch_wq4t(x, qweight, nullptr, scales, qzeros, nullptr, y, M, K, N, group_size,
                                        act_bf16, flags, static_cast<cudaStream_t>(stream));
      if (e != cudaErrorNotSupported) return from_cuda(e);
    }
    return from_cuda(launch_wq4_mma(x, qweight, scales, qzeros, y, M, K, N, group_size, act_bf16, flags,
                                    static_cast<cudaStream_t>(stream)));
  }

  if (!g_idx && K % wq4t_unit_k() == 0 && group_size % wq4t_unit_k() == 0) {
    const cudaError_t e = launch_wq4t(x, qweight, nullptr, scales, qzeros, nullptr, y, M, K, N, group_size, act_bf16,
                                      flags, static_cast<cudaStream_t>(stream));
    if (e != cudaErrorNotSupported) return from_cuda(e);
  }
  if (!g_idx && M >= 2 && group_size % wq4m_unit_k() == 0)
    return wq4m_launch(x, qweight, scales, qzeros, nullptr, y, M, K, N, group_size, act_bf16, flags,
                       static_cast<cudaStream_t>(stream));

  const int T = (N + 127) / 128, units = K / 32;
  LaunchPlan p{T, plan_splits(T, units), round_mt(M), flags, static_cast<cudaStream_t>(stream)};
  GemvArgs a{x, y, scales, qzeros, g_idx, M, K, N, group_size, 0};
  const bool act_order = g_idx != nullptr;
  a.ng_max = act_order ? 1 : max_groups_per_slice(units, p.S, 32, group_size);
  if (wq4_gemv_smem_bytes(p.MT, a.ng_max, act_order, K / group_size, p.S) > static_cast<size_t>(device_max_smem()))
    return WQ_ERR_UNSUPPORTED;
  CUtensorMap wmap, xmap, gmap;
  if (!encode_tensor_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, qweight, N, K / 8, size_t(N) * 4, 128, 32,
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_x_map(&xmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, x, K, M, 2, wq4_stage_k(), p.MT) ||
      (act_order && !encode_x_map(&gmap, CU_TENSOR_MAP_DATA_TYPE_INT32, g_idx, K, 1, 4, wq4_stage_k(), 1)))
    return WQ_ERR_CUDA;
  return from_cuda(launch_wq4_gemv(p, wmap, xmap, act_order ? &gmap : nullptr, a, act_bf16, qzeros != nullptr));
}

WQ_API wq_status wq4_actorder_prepare(const int32_t* qweight, const int32_t* g_idx, int K, int N, int group_size,
                                      int32_t* qweight_sorted, int32_t* perm, void* stream) {
  if (!qweight || !g_idx || !qweight_sorted || !perm) return WQ_ERR_NULL;
  if (K < 32 || N < 1 || K > kMaxDim || N > kMaxDim) return WQ_ERR_SHAPE;
  if (group_size < 32 || group_size % 32 != 0 || K % group_size != 0 || N % 8 != 0) return WQ_ERR_SHAPE;
  if (!aligned16(qweight) || !aligned16(g_idx) || !aligned16(qweight_sorted) || !aligned16(perm)) return WQ_ERR_ALIGN;
  const int r = actorder_prepare(qweight, g_idx, K, N, group_size, qweight_sorted, perm,
                                 static_cast<cudaStream_t>(stream));
  return r == 0 ? WQ_OK : (r == 1 ? WQ_ERR_SHAPE : WQ_ERR_CUDA);
}

WQ_API wq_status wq4_gemm_sorted(const void* x, const int32_t* qweight_sorted, const void* scales,
                                 const int32_t* qzeros, const int32_t* perm, void* y, int M, int K, int N,
                                 int group_size, int act_dtype, unsigned flags, void* stream) {
  if (!x || !qweight_sorted || !scales || !perm || !y) return WQ_ERR_NULL;
  if (M < 1 || M > 8 || K < 32 || N < 1 || K > kMaxDim || N > kMaxDim) return WQ_ERR_SHAPE;
  if (group_size < 32 || group_size % 32 != 0 || K % group_size != 0 || N % 8 != 0) return WQ_ERR_SHAPE;
  if (act_dtype != WQ_F16 && act_dtype != WQ_BF16) return WQ_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(qweight_sorted) || !aligned16(scales) || !aligned16(perm) || !aligned16(y) ||
      (qzeros && !aligned16(qzeros)))
    return WQ_ERR_ALIGN;
  if (K % wq4t_unit_k() == 0 && group_size % wq4t_unit_k() == 0) {
    const cudaError_t e = launch_wq4t(x, qweight_sorted, nullptr, scales, qzeros, perm, y, M, K, N, group_size,
                                      act_dtype == WQ_BF16, flags, static_cast<cudaStream_t>(stream));
    if (e != cudaErrorNotSupported) return from_cuda(e);
  }
  if (M >= 2 && group_size % wq4m_unit_k() == 0)
    return wq4m_launch(x, qweight_sorted, scales, qzeros, perm, y, M, K, N, group_size, act_dtype == WQ_BF16, flags,
                       static_cast<cudaStream_t>(stream));
  const int T = (N + 127) / 128, units = K / 32;
  LaunchPlan p{T, plan_splits(T, units), round_mt(M), flags, static_cast<cudaStream_t>(stream)};
  GemvArgs a{x, y, scales, qzeros, nullptr, M, K, N, group_size, 0};
  a.ng_max = max_groups_per_slice(units, p.S, 32, group_size);
  if (wq4_gemv_smem_bytes(p.MT, a.ng_max, false, 0, p.S, size_t(p.MT) * K * 2) > static_cast<size_t>(device_max_smem()))
    return WQ_ERR_UNSUPPORTED;
  CUtensorMap wmap, pmap;
  if (!encode_tensor_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, qweight_sorted, N, K / 8, size_t(N) * 4, 128, 32,
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_x_map(&pmap, CU_TENSOR_MAP_DATA_TYPE_INT32, perm, K, 1, 4, wq4_stage_k(), 1))
    return WQ_ERR_CUDA;
  return from_cuda(launch_wq4_gemv(p, wmap, pmap, nullptr, a, act_dtype == WQ_BF16, qzeros != nullptr, true));
}

WQ_API wq_status wq4_repack_tiled(const int32_t* qweight, const int32_t* g_idx, int K, int N, int group_size,
                                  int32_t* qweight_tiled, int32_t* perm, void* stream) {
  if (!qweight || !qweight_tiled || (g_idx && !perm)) return WQ_ERR_NULL;
  if (K < 64 || N < 32 || K > kMaxDim || N > kMaxDim) return WQ_ERR_SHAPE;
  if (K % 64 != 0 || N % 32 != 0 || group_size < 64 || group_size % 64 != 0 || K % group_size != 0)
    return WQ_ERR_SHAPE;
  if (!aligned16(qweight) || !aligned16(qweight_tiled) || (g_idx && (!aligned16(g_idx) || !aligned16(perm))))
    return WQ_ERR_ALIGN;
  const int r = repack_tiled(qweight, g_idx, K, N, group_size, qweight_tiled, g_idx ? perm : nullptr,
                             static_cast<cudaStream_t>(stream));
  return r == 0 ? WQ_OK : (r == 1 ? WQ_ERR_SHAPE : WQ_ERR_CUDA);
}

WQ_API wq_status wq4_gemm_tiled(const void* x, const int32_t* qweight_tiled, const void* scales,
                                const int32_t* qzeros, const int32_t* perm, void* y, int M, int K, int N,
                                int group_size, int act_dtype, unsigned flags, void* stream) {
  if (!x || !qweight_tiled || !scales || !y) return WQ_ERR_NULL;
  if (M < 1 || M > 8 || K < 64 || N < 32 || K > kMaxDim || N > kMaxDim) return WQ_ERR_SHAPE;
  if (K % 64 != 0 || N % 32 != 0 || group_size < 64 || group_size % 64 != 0 || K % group_size != 0)
    return WQ_ERR_SHAPE;
  if (act_dtype != WQ_F16 && act_dtype != WQ_BF16) return WQ_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(qweight_tiled) || !aligned16(scales) || !aligned16(y) ||
      (qzeros && !aligned16(qzeros)) || (perm && !aligned16(perm)))
    return WQ_ERR_ALIGN;
  return from_cuda(launch_wq4t(x, nullptr, reinterpret_cast<const uint8_t*>(qweight_tiled), scales, qzeros, perm, y,
                               M, K, N, group_size, act_dtype == WQ_BF16, flags, static_cast<cudaStream_t>(stream)));
}

WQ_API wq_status wq8_dequant(const int8_t* w, const float* scales, float* w_out, int K, int N, int group_size,
                             unsigned flags, void* stream) {
  if (!w || !scales || !w_out) return WQ_ERR_NULL;
  if (K < 1 || N < 1 || K > kMaxDim || N > kMaxDim) return WQ_ERR_SHAPE;
  if (group_size < 16 || group_size % 16 != 0 || K % group_size != 0 || N % 16 != 0) return WQ_ERR_SHAPE;
  if (!aligned16(w) || !aligned16(scales) || !aligned16(w_out)) return WQ_ERR_ALIGN;
  return from_cuda(launch_wq8_dequant(w, scales, w_out, K, N, group_size, flags, static_cast<cudaStream_t>(stream)));
}

WQ_API wq_status wq3_dequant(const int32_t* mat, const void* scales, const void* zeros, void* w_out, int K, int N,
                             unsigned flags, void* stream) {
  if (!mat || !scales || !zeros || !w_out) return WQ_ERR_NULL;
  if (K < 32 || N < 1 || K > kMaxDim || N > kMaxDim) return WQ_ERR_SHAPE;
  if (K % 32 != 0 || N % 8 != 0) return WQ_ERR_SHAPE;
  if (!aligned16(mat) || !aligned16(scales) || !aligned16(zeros) || !aligned16(w_out)) return WQ_ERR_ALIGN;
  return from_cuda(launch_wq3_dequant(mat, scales, zeros, w_out, K, N, flags, static_cast<cudaStream_t>(stream)));
}

WQ_API wq_status wq4_dequant(const int32_t* qweight, const void* scales, const int32_t* qzeros,
                             const int32_t* g_idx, void* w_out, int K, int N, int group_size, int act_dtype,
                             unsigned flags, void* stream) {
  if (!qweight || !scales || !w_out) return WQ_ERR_NULL;
  if (K < 32 || N < 1 || K > kMaxDim || N > kMaxDim) return WQ_ERR_SHAPE;
  if (group_size < 32 || group_size % 32 != 0 || K % group_size != 0 || N % 8 != 0) return WQ_ERR_SHAPE;
  if (act_dtype != WQ_F16 && act_dtype != WQ_BF16) return WQ_ERR_UNSUPPORTED;
  if (!aligned16(qweight) || !aligned16(scales) || !aligned16(w_out) || (qzeros && !aligned16(qzeros)) ||
      (g_idx && !aligned16(g_idx)))
    return WQ_ERR_ALIGN;
  return from_cuda(launch_wq4_dequant(qweight, scales, qzeros, g_idx, w_out, K, N, group_size,
                                      act_dtype == WQ_BF16, flags, static_cast<cudaStream_t>(stream)));
}

WQ_API size_t w8a8_gemm_workspace_bytes(int M, int K, int N) { return w8a8_workspace_bytes(M, K, N); }

WQ_API wq_status w8a8_gemm(const void* X, const int8_t* W, const float* Sw, void* Y, int M, int K, int N,
                           int8_t* Xq_out, float* Sx_out, int32_t* acc_out, void* workspace,
                           size_t workspace_bytes, unsigned flags, void* stream) {
  if (!X || !W || !Sw || !Y || !workspace) return (!workspace && X && W && Sw && Y) ? WQ_ERR_WORKSPACE : WQ_ERR_NULL;
  if (M < 1 || K < 64 || N < 16 || M > kMaxDim || K > 65536 || N > kMaxDim) return WQ_ERR_SHAPE;
  if (K % 64 != 0 || N % 16 != 0) return WQ_ERR_SHAPE;
  if (!aligned16(X) || !aligned16(W) || !aligned16(Sw) || !aligned16(Y) || (Xq_out && !aligned16(Xq_out)) ||
      (Sx_out && !aligned16(Sx_out)) || (acc_out && !aligned16(acc_out)) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return WQ_ERR_ALIGN;
  if (workspace_bytes < w8a8_workspace_bytes(M, K, N)) return WQ_ERR_WORKSPACE;
  return from_cuda(launch_w8a8(X, W, Sw, Y, M, K, N, Xq_out, Sx_out, acc_out, workspace, flags,
                               static_cast<cudaStream_t>(stream)));
}

WQ_API wq_status w8a8_gemm_smooth(const void* X, const float* smooth, const int8_t* W, const float* Sw, void* Y,
                                  int M, int K, int N, int8_t* Xq_out, float* Sx_out, int32_t* acc_out,
                                  void* workspace, size_t workspace_bytes, unsigned flags, void* stream) {
  if (!smooth) return WQ_ERR_NULL;
  if (!aligned16(smooth)) return WQ_ERR_ALIGN;
  if (!X || !W || !Sw || !Y || !workspace) return (!workspace && X && W && Sw && Y) ? WQ_ERR_WORKSPACE : WQ_ERR_NULL;
  if (M < 1 || K < 64 || N < 16 || M > kMaxDim || K > 65536 || N > kMaxDim) return WQ_ERR_SHAPE;
  if (K % 64 != 0 || N % 16 != 0) return WQ_ERR_SHAPE;
  if (!aligned16(X) || !aligned16(W) || !aligned16(Sw) || !aligned16(Y) || (Xq_out && !aligned16(Xq_out)) ||
      (Sx_out && !aligned16(Sx_out)) || (acc_out && !aligned16(acc_out)) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return WQ_ERR_ALIGN;
  if (workspace_bytes < w8a8_workspace_bytes(M, K, N)) return WQ_ERR_WORKSPACE;
  return from_cuda(launch_w8a8(X, W, Sw, Y, M, K, N, Xq_out, Sx_out, acc_out, workspace, flags,
                               static_cast<cudaStream_t>(stream), smooth));
}

WQ_API size_t w8a8_gemm_outlier_workspace_bytes(int M, int K, int N) { return w8a8_outlier_workspace_bytes(M, K, N); }

WQ_API wq_status w8a8_gemm_outlier(const void* X, const int8_t* W, const float* Sw, void* Y, int M, int K, int N,
                                   float threshold, int8_t* Xq_out, float* Sx_out, int32_t* acc_out,
                                   int32_t* n_outliers_out, void* workspace, size_t workspace_bytes, unsigned flags,
                                   void* stream) {
  if (!X || !W || !Sw || !Y || !workspace) return (!workspace && X && W && Sw && Y) ? WQ_ERR_WORKSPACE : WQ_ERR_NULL;
  if (M < 1 || K < 64 || N < 16 || M > kMaxDim || K > 65536 || N > kMaxDim) return WQ_ERR_SHAPE;
  if (K % 64 != 0 || N % 16 != 0) return WQ_ERR_SHAPE;
  if (!aligned16(X) || !aligned16(W) || !aligned16(Sw) || !aligned16(Y) || (Xq_out && !aligned16(Xq_out)) ||
      (Sx_out && !aligned16(Sx_out)) || (acc_out && !aligned16(acc_out)) ||
      (n_outliers_out && (reinterpret_cast<uintptr_t>(n_outliers_out) & 3u) != 0) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return WQ_ERR_ALIGN;
  if (workspace_bytes < w8a8_outlier_workspace_bytes(M, K, N)) return WQ_ERR_WORKSPACE;
  return from_cuda(launch_w8a8(X, W, Sw, Y, M, K, N, Xq_out, Sx_out, acc_out, workspace, flags,
                               static_cast<cudaStream_t>(stream), nullptr, &threshold, n_outliers_out));
}

}  // extern "C"
