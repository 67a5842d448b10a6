// w8a8.cu -- W8A8 dynamic-quantization GEMM on the tcgen05 tensor cores.
//
// Definition ("Quantization CUDA", Dynamic Quantization and 优化):
//   Sx[m]    = fp32(max_k |X[m,k]| / 127)          (activations quantized at run time, per token)
//   Xq[m,k]  = clamp(rint(fp32(X[m,k] / Sx[m])), -127, 127)
//   acc[m,n] = sum_k Xq[m,k] * W[k,n]              (int8 multiply, exact int32 accumulate)
//   Y[m,n]   = bf16(Sx[m] * acc[m,n] * Sw[n])      (rescale fused into the matmul epilogue)
//
// sm_103a has no integer tcgen05 MMA, so the product runs as kind::f16 on
// fp16 operands that hold the integer codes exactly (X codes in [-127, 127],
// weights in [-128, 127]).  Every
// product is an exact integer and so is every partial sum below 2^24: the
// tensor core accumulates 256 values of k (|sum| <= 256 * 127 * 128 < 2^22) into
// an fp32 tensor-memory accumulator, and the epilogue warps fold each such
// chunk into an int32 register sum with the magic-number conversion
// bits(f + 1.5 * 2^23) (exact for |f| < 2^22; the constant is removed once at
// the end, in wrapping unsigned arithmetic).  The int32 result is never
// stored unless a debug output is requested.
//
// Kernels: (0) LLM.int8() only: w8a8_outlier_scan_kernel flags the columns of
// X holding a value above the threshold, w8a8_outlier_compact_kernel lists
// them; (1) w8a8_quant_kernel, one CTA per row: Sx, the int8 codes (if
// requested) and fp16 copies of the codes in the workspace, after the optional
// Smoothquant division and with LLM.int8()'s outlier columns zeroed; (2)
// w8a8_mma_kernel, one 128 x 128 output tile per CTA, 128-value k stages:
//   warp 16 : TMA of the int8 W tile (lane 0, before the dependency wait) and
//             of the fp16 X code tile (lane 1), both 128-byte swizzled;
//   warps 0-7 : convert the int8 W tile to fp16 (exact) and store it
//             transposed into tensor memory, where it is the A operand;
//   warp 17 : eight MMAs (M = N = 128, K = 16) per stage, A from tensor
//             memory, B = X from shared memory, into one of two tensor-memory
//             accumulators (one per 256-value chunk of k);
//   warps 8-15 : drain each chunk into int32 and, at the end, write
//             Y = bf16(Sx * acc * Sw) through shared memory with coalesced stores
//             (the LLM.int8() instance adds the outlier columns' 16-bit product
//             in fp32 first).
#include <algorithm>

#include "../../include/wq.h"
#include "wq_gemv_common.cuh"
#include "wq_mma.h"
#include "wq_tcgen05.cuh"

namespace wq {

bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swizzle);
int device_max_smem();

namespace {

// ------------------------------------------------------------ quantization --
// smooth (fp32 [K] or null): Smoothquant's per-channel divisor ("Quantization
// CUDA", Smoothquant: Y = (X diag(s)^-1)(diag(s) W)); every activation is
// divided by it (one correctly rounded fp32 division) before the row amax and
// the codes.
// out_flags (int [K] or null): LLM.int8()'s outlier columns, quantized as zero
// here (their product runs in 16-bit floating point in the GEMM epilogue).
__global__ void __launch_bounds__(256) w8a8_quant_kernel(const uint16_t* __restrict__ X, int K,
                                                         const float* __restrict__ smooth,
                                                         const int* __restrict__ out_flags,
                                                         __half* __restrict__ xq16, float* __restrict__ sx_ws,
                                                         int8_t* __restrict__ xq_out, float* __restrict__ sx_out) {
  __shared__ float red[8];
  const int m = blockIdx.x;
  pdl_wait();
  const uint16_t* row = X + size_t(m) * K;
  float amax = 0.f;
  // the 8 activations k .. k+7 of this row, divided by the smoothing factors if any
  auto load8 = [&](int k, float (&x)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = bf16_bits_to_f32((i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu));
    if (smooth) {
      const float4 s0 = *reinterpret_cast<const float4*>(smooth + k);
      const float4 s1 = *reinterpret_cast<const float4*>(smooth + k + 4);
      const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = __fdiv_rn(x[i], sv[i]);
    }
    if (out_flags) {
      const int4 f0 = *reinterpret_cast<const int4*>(out_flags + k);
      const int4 f1 = *reinterpret_cast<const int4*>(out_flags + k + 4);
      const int fv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = fv[i] ? 0.f : x[i];
    }
  };
  for (int k = threadIdx.x * 8; k < K; k += 256 * 8) {
    float x[8];
    load8(k, x);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float sx = __fdiv_rn(amax, 127.0f);
  for (int k = threadIdx.x * 8; k < K; k += 256 * 8) {
    float x[8];
    load8(k, x);
    int q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int c = 0;
      if (sx != 0.f) c = min(127, max(-127, __float2int_rn(__fdiv_rn(x[i], sx))));
      q[i] = c;
    }
    // fp16 copies in the GEMM's operand order: k0 + {0,2}, {4,6}, {1,3}, {5,7}
    uint4 h;
    h.x = uint32_t(__half_as_ushort(__int2half_rn(q[0]))) | (uint32_t(__half_as_ushort(__int2half_rn(q[2]))) << 16);
    h.y = uint32_t(__half_as_ushort(__int2half_rn(q[4]))) | (uint32_t(__half_as_ushort(__int2half_rn(q[6]))) << 16);
    h.z = uint32_t(__half_as_ushort(__int2half_rn(q[1]))) | (uint32_t(__half_as_ushort(__int2half_rn(q[3]))) << 16);
    h.w = uint32_t(__half_as_ushort(__int2half_rn(q[5]))) | (uint32_t(__half_as_ushort(__int2half_rn(q[7]))) << 16);
    *reinterpret_cast<uint4*>(xq16 + size_t(m) * K + k) = h;
    if (xq_out) {
      uint2 b;
      b.x = (uint32_t(q[0]) & 0xFFu) | ((uint32_t(q[1]) & 0xFFu) << 8) | ((uint32_t(q[2]) & 0xFFu) << 16) |
            ((uint32_t(q[3]) & 0xFFu) << 24);
      b.y = (uint32_t(q[4]) & 0xFFu) | ((uint32_t(q[5]) & 0xFFu) << 8) | ((uint32_t(q[6]) & 0xFFu) << 16) |
            ((uint32_t(q[7]) & 0xFFu) << 24);
      *reinterpret_cast<uint2*>(xq_out + size_t(m) * K + k) = b;
    }
  }
  if (threadIdx.x == 0) {
    sx_ws[m] = sx;
    if (sx_out) sx_out[m] = sx;
  }
  pdl_launch_dependents();  // the GEMM may start once every row's codes are written
}

// --------------------------------------------------------- LLM.int8() scan --
// ("Quantization CUDA", LLM.int8(): the activation columns holding a value
// above the threshold, with the matching weight rows, are multiplied in 16-bit
// floating point.)  flags[k] = 1 when some |X[m,k]| > threshold: one thread
// covers 8 columns (one 16-byte load per row) over a chunk of kScanRows rows,
// all loads in flight at once.
constexpr int kScanRows = 8;
__global__ void __launch_bounds__(256) w8a8_outlier_scan_kernel(const uint16_t* __restrict__ X, int M, int K,
                                                                float threshold, int* __restrict__ flags) {
  pdl_launch_dependents();
  pdl_wait();
  const int k = (blockIdx.x * 256 + threadIdx.x) * 8;
  if (k >= K) return;
  uint32_t hit = 0;  // bit i: column k + i
  for (int m0 = blockIdx.y * kScanRows; m0 < M; m0 += gridDim.y * kScanRows) {  // grid-stride over row chunks
    uint4 rows[kScanRows];
#pragma unroll
    for (int j = 0; j < kScanRows; ++j)
      rows[j] = (m0 + j < M) ? *reinterpret_cast<const uint4*>(X + size_t(m0 + j) * K + k) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < kScanRows; ++j) {
      const uint32_t w[4] = {rows[j].x, rows[j].y, rows[j].z, rows[j].w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (fabsf(bf16_bits_to_f32((i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu))) > threshold) hit |= 1u << i;
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if ((hit >> i) & 1u) flags[k + i] = 1;
}

// The outlier columns of X, transposed: xoT[j][m] = X[m, idx[j]] (raw bf16),
// gathered once per call so that the GEMM epilogue of every column tile reads
// each outlier column of its rows as one contiguous run instead of one
// scattered 2-byte load per element and tile.  One thread per row m.
__global__ void __launch_bounds__(256) w8a8_outlier_gather_kernel(const uint16_t* __restrict__ X, int M, int K,
                                                                  const int* __restrict__ idx,
                                                                  const int* __restrict__ count,
                                                                  uint16_t* __restrict__ xoT) {
  pdl_launch_dependents();
  pdl_wait();
  const int m = blockIdx.x * 256 + threadIdx.x;
  if (m >= M) return;
  const int cnt = *count;
  for (int j = 0; j < cnt; ++j) xoT[size_t(j) * M + m] = X[size_t(m) * K + idx[j]];
}

// The flagged columns in increasing order (idx) and their number (count, and
// *count_out when given): one CTA, a block-wide exclusive scan of per-thread counts.
__global__ void __launch_bounds__(1024) w8a8_outlier_compact_kernel(const int* __restrict__ flags, int K,
                                                                    int* __restrict__ idx, int* __restrict__ count,
                                                                    int* __restrict__ count_out) {
  __shared__ int warp_sum[32];
  pdl_launch_dependents();
  pdl_wait();
  const int per = (K + 1023) / 1024;
  const int k0 = min(K, int(threadIdx.x) * per), k1 = min(K, k0 + per);
  int c = 0;
  for (int k = k0; k < k1; ++k) c += flags[k] != 0;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = c;  // inclusive scan within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_sum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int v = warp_sum[lane], wincl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wincl, o);
      if (lane >= o) wincl += t;
    }
    warp_sum[lane] = wincl - v;  // exclusive prefix of the warp totals
  }
  __syncthreads();
  int pos = warp_sum[wid] + incl - c;
  for (int k = k0; k < k1; ++k)
    if (flags[k]) idx[pos++] = k;
  if (threadIdx.x == blockDim.x - 1) {
    *count = pos;
    if (count_out) *count_out = pos;
  }
}

// --------------------------------------------------------------------- GEMM --
// Roles: the tensor core computes D[n, m] = sum_k W[k, n] X[m, k] for a tile of
// 128 columns n (MMA M, operand A = W^T in tensor memory) by 128 rows m (MMA N,
// operand B = the fp16 X codes in shared memory, K-major).  W reaches tensor
// memory straight from registers, so its fp16 copy never passes through shared
// memory: shared memory carries only the TMA writes of both tiles, the
// converters' reads of the int8 W tile and the MMA's reads of X.
constexpr int kBM = 128, kBN = 128, kBK = 128;
constexpr int kBoxK = 64;                    // values of k per 128-byte-swizzled X box
constexpr int kChunkStages = 256 / kBK;      // 256 values of k per exact fp32 chunk
// A stage slot s holds the fp16 X codes (shared memory) and the fp16 W^T
// (tensor memory) of one stage; both are released by one MMA commit.
constexpr int kNS = 4;
constexpr int kNSW = 4;                      // int8 W shared-memory ring
constexpr int kConvGroups = 2;               // converter groups take alternate stages
constexpr int kConvWarps = 4 * kConvGroups;  // one warp per tensor-memory lane quarter and group
constexpr int kEpiWarps = 8;             // two per tensor-memory lane quarter, 64 columns each
constexpr int kThreads = (kConvWarps + kEpiWarps + 2) * 32;
constexpr int kWarpTMA = kConvWarps + kEpiWarps, kWarpMMA = kWarpTMA + 1;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kEpiCols = kBM / (kEpiWarps / 4);  // accumulator columns (rows m) per epilogue thread
constexpr int kXBoxBytes = kBM * kBoxK * 2;  // 16 KB: one X box (128 rows x 64 k)
constexpr int kXBytes = kBM * kBK * 2;       // 32 KB fp16 codes of X per stage (two boxes)
constexpr int kWBytes = kBK * kBN;           // 16 KB int8 W per stage (128-byte swizzle)
constexpr uint32_t kDCols = kBM;             // fp32 accumulator columns per buffer
constexpr uint32_t kACols = kBK / 2;         // 64 columns of fp16 pairs per W^T stage
constexpr uint32_t kTmemCols = 2 * kDCols + kNS * kACols;  // 512
constexpr int kOutStride = kBN * 2 + 16;     // padded bf16 output row in shared memory
constexpr int kOutChunk = 32;                // outlier columns staged per round (LLM.int8())
constexpr int kOutlierStage = 64 * 1024;     // their x [128 m][32] and w [32][128 n] fp32, in the X ring
static_assert(kTmemCols <= 512, "tensor memory holds 512 columns");
static_assert(kEpiCols == 64, "the epilogue loop reads 16-column groups of a 64-column half");

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) & ~(a - 1); }

struct SmemW8A8 {
  size_t x, w, sx, pre, bars, misc, total;
  __host__ __device__ SmemW8A8() {
    size_t o = 0;
    x = o;    o += size_t(kNS) * kXBytes;     // also the output staging area at the end
    w = o;    o += size_t(kNSW) * kWBytes;
    sx = o;   o = align_up(o + kBM * 4, 16);
    pre = o;  o = align_up(o + size_t(kOutChunk) * (kBM * 2 + kBN), 16);  // LLM.int8(): first outlier chunk
    bars = o; o = align_up(o + size_t(2 * kNS + 2 * kNSW + 4) * 8, 16);
    misc = o; o = align_up(o + 32, 16);
    total = o + 1024;
  }
};
static_assert(kBM * kOutStride <= kNS * kXBytes, "the output tile is staged in the X ring");
static_assert(kBM * kOutStride <= kOutlierStage &&
                  kOutlierStage + (kBM + kBN + 1) * kOutChunk * 4 <= kNS * kXBytes,
              "the outlier operands sit in the X ring after the output staging area");
static_assert(kNS % kConvGroups == 0, "a stage slot is always refilled by the same converter group");

struct W8A8Args {
  const float* Sw;
  const float* Sx;       // workspace copy written by the quantization kernel
  void* Y;
  int32_t* acc_out;
  // LLM.int8() (all null otherwise): the outlier columns and their number, the
  // gathered bf16 activations of those columns (xoT [count][M]) and the int8
  // weights their 16-bit product reads
  const int* out_idx;
  const int* out_count;
  const uint16_t* XoT;
  const int8_t* Wb;
  int M, K, N;
};

// 4 x 4 byte transpose across the lanes 4i .. 4i + 3 of a warp: lane 4i + j
// holds word w_j (4 bytes, one per column) and ends with byte j of w_0 .. w_3.
// Two exchange rounds (lane ^ 2, then lane ^ 1), one byte permute each.
__device__ __forceinline__ uint32_t quad_transpose(uint32_t w, uint32_t sel1, uint32_t sel2) {
  const uint32_t y = prmt(w, __shfl_xor_sync(0xffffffffu, w, 2), sel1);
  return prmt(y, __shfl_xor_sync(0xffffffffu, y, 1), sel2);
}

// OUTLIER: the LLM.int8() epilogue (a separate instance, so that the plain
// GEMM carries none of its code or registers).
template <bool OUTLIER>
__global__ void __launch_bounds__(kThreads, 1)
    w8a8_mma_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                    const W8A8Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemW8A8 L;
  uint8_t* sX = smem + L.x;
  uint8_t* sW = smem + L.w;
  float* sSx = reinterpret_cast<float*>(smem + L.sx);
  // full / empty: stage slots (X codes landed and W^T stored / both read by the MMAs);
  // wfull / wempty: the int8 W ring (released as soon as the converters have read it);
  // t_full / t_empty: the two accumulator buffers (one per 256-value chunk of k)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kNS;
  uint64_t* wfull = empty + kNS;
  uint64_t* wempty = wfull + kNSW;
  uint64_t* t_full = wempty + kNSW;
  uint64_t* t_empty = t_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L.misc + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM;
  const int M = a.M, K = a.K, N = a.N;
  const int nst = (K + kBK - 1) / kBK;  // the tail of the last stage is zero-filled by TMA
  const int nchunks = (nst + kChunkStages - 1) / kChunkStages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&full[s], 4 + 1);  // the four converter warps of a group, and the X producer (with bytes)
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kNSW; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&t_full[s], 1);
      mbar_init(&t_empty[s], kEpiWarps);
    }
    *failed = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_a = tmem + 2 * kDCols;  // first column of the W^T stages
  pdl_launch_dependents();

  if (warp == kWarpTMA) {
    // ------------------------------------------------------------ producer --
    // lane 0 streams the int8 W tiles (weight-side data: no dependency wait, the
    // converters can start before the previous kernel has finished); lane 1
    // streams the fp16 X codes after the wait.
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      for (int i = 0; i < nst && !*failed; ++i) {
        const int s = i % kNSW;
        if (i >= kNSW && !mbar_wait_sleep(&wempty[s], ((i / kNSW) - 1) & 1)) {
          *failed = 1;
          break;
        }
        mbar_expect_tx(&wfull[s], kWBytes);
        tma_load_2d(sW + size_t(s) * kWBytes, &wmap, &wfull[s], n0, i * kBK, 0ull);
      }
    } else if (lane == 1) {
      prefetch_tensormap(&xmap);
      pdl_wait();
      for (int i = 0; i < nst && !*failed; ++i) {
        const int s = i % kNS;
        if (i >= kNS && !mbar_wait_sleep(&empty[s], ((i / kNS) - 1) & 1)) {
          *failed = 1;
          break;
        }
        mbar_expect_tx(&full[s], kXBytes);
#pragma unroll
        for (int h = 0; h < kBK / kBoxK; ++h)
          tma_load_2d(sX + size_t(s) * kXBytes + h * kXBoxBytes, &xmap, &full[s], i * kBK + h * kBoxK, m0, 0ull);
      }
    } else {
      pdl_wait();
    }
  } else if (warp == kWarpMMA) {
    // ----------------------------------------------------------------- MMA --
    pdl_wait();
    if (lane == 0) {
      constexpr uint32_t idesc = f16_idesc(kBN, kBM, 0);  // M = 128 columns n, N = 128 rows m, fp16, fp32 acc
      int last = -1;
      for (int i = 0; i < nst; ++i) {
        const int s = i % kNS, ch = i / kChunkStages, tb = ch & 1;
        if (i % kChunkStages == 0 && ch >= 2) {
          if (!mbar_wait_sleep(&t_empty[tb], ((ch / 2) - 1) & 1)) { *failed = 1; break; }
        }
        if (!mbar_wait_sleep(&full[s], (i / kNS) & 1)) {
          *failed = 1;
          break;
        }
        tc_fence_after();
        const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sX + size_t(s) * kXBytes));
        const uint32_t acol = tmem_a + s * kACols;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_f16_ts(tmem + tb * kDCols, acol + 8 * k,
                     bdesc + uint64_t(((k / (kBoxK / 16)) * kXBoxBytes + 32 * (k % (kBoxK / 16))) >> 4), idesc,
                     (i % kChunkStages != 0 || k > 0) ? 1u : 0u);
        mma_commit(&empty[s]);
        if (i % kChunkStages == kChunkStages - 1 || i == nst - 1) mma_commit(&t_full[tb]);
        last = i;
      }
      if (last >= 0) mbar_wait_sleep(&empty[last % kNS], (last / kNS) & 1);
    }
  } else if (warp < kConvWarps) {
    // ---------------------------------------------------------- converters --
    // Warp c writes tensor-memory lanes 32 (c % 4) .. (columns n of the tile)
    // of the stages i with i % kConvGroups == c / 4.  Per block of 8 values of
    // k, lane 4i + j reads 4 bytes (columns 32 (c % 4) + 4i ..) of rows k0 + 2j
    // (word A) and k0 + 2j + 1 (word B) of the swizzled int8 tile; a 4 x 4
    // transpose across the lane quad leaves lane l with column 32 (c % 4) + l of
    // rows k0, k0+2, k0+4, k0+6 (A) and k0+1, k0+3, k0+5, k0+7 (B).  Each byte
    // b = q + 128 becomes the fp16 1024 + b and then q exactly.  The columns of
    // fp16 pairs hold k0 + {0,2}, {4,6}, {1,3}, {5,7}: the quantization kernel
    // stores the X codes of every 8-value block in that order.
    const int quarter = warp & 3, group = warp >> 2;
    const int qi = lane >> 2, qj = lane & 3;
    const uint32_t sel1 = (qj & 2) ? 0x3276u : 0x5410u;
    const uint32_t sel2 = (qj & 1) ? 0x3715u : 0x6240u;
    const int chunk = 2 * quarter + (qi >> 2), cbyte = 4 * (qi & 3);
    const int offa = ((chunk ^ (2 * qj)) << 4) + cbyte, offb = ((chunk ^ (2 * qj + 1)) << 4) + cbyte;
    const uint32_t taddr = tmem_a + (static_cast<uint32_t>(quarter * 32) << 16);
    for (int i = group; i < nst; i += kConvGroups) {
      const int s = i % kNS, ws = i % kNSW;
      // warp-uniform decisions: the shuffles and tensor-memory stores below need the whole warp
      if (!__all_sync(0xffffffffu, mbar_wait_sleep(&wfull[ws], (i / kNSW) & 1))) { *failed = 1; break; }
      if (i >= kNS && !__all_sync(0xffffffffu, mbar_wait_sleep(&empty[s], ((i / kNS) - 1) & 1))) { *failed = 1; break; }
      tc_fence_after();
      const uint8_t* wt = sW + size_t(ws) * kWBytes + 2 * qj * kBN;
      uint32_t h[kACols];
#pragma unroll
      for (int b = 0; b < kBK / 8; ++b) {
        uint32_t wa = *reinterpret_cast<const uint32_t*>(wt + 8 * b * kBN + offa);       // row 8b + 2 qj
        uint32_t wb = *reinterpret_cast<const uint32_t*>(wt + (8 * b + 1) * kBN + offb); // row 8b + 2 qj + 1
        wa = quad_transpose(wa, sel1, sel2) ^ 0x80808080u;
        wb = quad_transpose(wb, sel1, sel2) ^ 0x80808080u;
        const uint32_t p[4] = {prmt(wa, 0x64646464u, 0x4140u), prmt(wa, 0x64646464u, 0x4342u),
                               prmt(wb, 0x64646464u, 0x4140u), prmt(wb, 0x64646464u, 0x4342u)};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(h[4 * b + j]) : "r"(p[j]), "r"(0x64806480u));
      }
      // one arrival per warp: many threads arriving on one barrier serialise
      __syncwarp();
      if (lane == 0) mbar_arrive(&wempty[ws]);  // the warp's reads of the W stage are done (values in registers)
      tmem_st32(taddr + s * kACols, h);
      tmem_st32(taddr + s * kACols + 32, h + 32);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[s]);
    }
    pdl_wait();
  } else {
    // ------------------------------------------------------------ epilogue --
    // warp e (0..7): tensor-memory lane quarter e % 4 = tile columns n
    // 32 (e % 4) .., accumulator columns (tile rows m) kEpiCols * (e / 4) ..
    pdl_wait();
    const int et = threadIdx.x - kConvThreads;  // 0 .. kEpiThreads - 1
    const int ew = warp - kConvWarps, quarter = ew & 3, half = ew >> 2;
    const int col = quarter * 32 + lane;            // tensor-memory lane == tile column n
    const int cbase = half * kEpiCols;
    const float sw = (n0 + col < N) ? a.Sw[n0 + col] : 0.f;
    for (int r = et; r < kBM; r += kEpiThreads) sSx[r] = (m0 + r < M) ? a.Sx[m0 + r] : 0.f;
    // LLM.int8(): the tile's share of the first kOutChunk outlier columns --
    // activations (bf16, [j][m]) and weight rows (int8, [j][n]) -- fetched now,
    // while the main loop runs: in the epilogue their three dependent global
    // loads (count, column list, values) cost ~1-2 us per tile under load
    uint16_t* pre_x = reinterpret_cast<uint16_t*>(smem + L.pre);
    int8_t* pre_w = reinterpret_cast<int8_t*>(pre_x + kOutChunk * kBM);
    const int cnt0 = OUTLIER ? min(kOutChunk, *a.out_count) : 0;
    if (OUTLIER) {
#pragma unroll 4
      for (int t = 0; t < kOutChunk * kBM / kEpiThreads; ++t) {
        const int i = et + t * kEpiThreads, j = i / kBM, m = i % kBM;  // j is the same across a warp
        if (j < cnt0) pre_x[i] = (m0 + m < M) ? a.XoT[size_t(j) * M + m0 + m] : uint16_t(0);
      }
#pragma unroll 4
      for (int t = 0; t < kOutChunk * kBN / kEpiThreads; ++t) {
        const int i = et + t * kEpiThreads, j = i / kBN, n = i % kBN;
        if (j < cnt0) pre_w[i] = (n0 + n < N) ? a.Wb[size_t(a.out_idx[j]) * N + n0 + n] : int8_t(0);
      }
    }
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + cbase;
    uint32_t acc[kEpiCols];
#pragma unroll
    for (int c = 0; c < kEpiCols; ++c) acc[c] = 0u;
    int drained = 0;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int tb = ch & 1;
      if (!__all_sync(0xffffffffu, mbar_wait_sleep(&t_full[tb], (ch / 2) & 1))) { *failed = 1; break; }
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < kEpiCols; c0 += 16) {
        float v[16];
        tmem_ld16(lane_addr + tb * kDCols + c0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[c0 + j] += __float_as_uint(v[j] + 12582912.0f);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&t_empty[tb]);
      ++drained;
    }
    const uint32_t bias = uint32_t(drained) * 0x4B400000u;
    // Y = bf16(Sx * acc * Sw) staged in shared memory (the X stages are free now:
    // the MMA warp saw the last one released before the epilogue's last chunk)
    asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");  // epilogue warps: sSx complete
    const bool col_ok = n0 + col < N;
    // the int32 product (debug output), then y = (Sx * acc) * Sw in fp32, in place
#pragma unroll
    for (int c = 0; c < kEpiCols; ++c) {
      const int r = cbase + c;
      const int32_t iv = static_cast<int32_t>(acc[c] - bias);
      if (a.acc_out && col_ok && m0 + r < M) a.acc_out[size_t(m0 + r) * N + n0 + col] = iv;
      acc[c] = __float_as_uint((sSx[r] * static_cast<float>(iv)) * sw);
    }
    if (OUTLIER) {
      // LLM.int8(): y += sum_j X[m, idx_j] * (Sw[n] * W[idx_j, n]) over the outlier
      // columns: the first kOutChunk prefetched, the rest staged kOutChunk at a
      // time in the (now free) X ring
      const int cnt = *a.out_count;
      float* xo = reinterpret_cast<float*>(sX + kOutlierStage);  // [kBM][kOutChunk]
      float* wo = xo + kBM * kOutChunk;                           // [kOutChunk][kBN]
      int* sidx = reinterpret_cast<int*>(wo + kOutChunk * kBN);   // [kOutChunk] column indices
      asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");  // the prefetched chunk is complete
      for (int j = 0; j < cnt0; ++j) {
        const float sww = sw * static_cast<float>(pre_w[j * kBN + col]);
#pragma unroll
        for (int c = 0; c < kEpiCols; ++c)
          acc[c] = __float_as_uint(fmaf(bf16_bits_to_f32(pre_x[j * kBM + cbase + c]), sww, __uint_as_float(acc[c])));
      }
      // further chunks (more than kOutChunk outlier columns): fetched here
      for (int j0 = kOutChunk; j0 < cnt; j0 += kOutChunk) {
        const int nj = min(kOutChunk, cnt - j0);
        asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");  // the previous round is consumed
        if (et < kOutChunk) sidx[et] = et < nj ? a.out_idx[j0 + et] : 0;
        asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");
        // the kBM x nj real activations spread over every thread, all loads in flight at once
        // (slots j >= nj are never read)
#pragma unroll
        for (int t = 0; t < kBM * kOutChunk / kEpiThreads; ++t) {
          const int i = et + t * kEpiThreads;
          if (i < kBM * nj) {
            const int m = i % kBM, j = i / kBM;  // consecutive threads, consecutive rows of one column
            xo[m * kOutChunk + j] = (m0 + m < M) ? bf16_bits_to_f32(a.XoT[size_t(j0 + j) * M + m0 + m]) : 0.f;
          }
        }
#pragma unroll
        for (int t = 0; t < kOutChunk * kBN / kEpiThreads; ++t) {
          const int i = et + t * kEpiThreads, j = i / kBN, n = i % kBN;
          wo[i] = (j < nj && n0 + n < N) ? static_cast<float>(a.Wb[size_t(sidx[j]) * N + n0 + n]) : 0.f;
        }
        asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");
        for (int j = 0; j < nj; ++j) {
          const float sww = sw * wo[j * kBN + col];
#pragma unroll
          for (int c = 0; c < kEpiCols; ++c)
            acc[c] = __float_as_uint(fmaf(xo[(cbase + c) * kOutChunk + j], sww, __uint_as_float(acc[c])));
        }
      }
    }
    uint16_t* ocol = reinterpret_cast<uint16_t*>(sX) + col;
#pragma unroll
    for (int c = 0; c < kEpiCols; ++c)
      ocol[size_t(cbase + c) * (kOutStride / 2)] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(acc[c])));
    asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");
    // coalesced stores: 16 chunks of 16 bytes per tile row
    uint16_t* Y = static_cast<uint16_t*>(a.Y);
    for (int q = et; q < kBM * (kBN / 8); q += kEpiThreads) {
      const int r = q / (kBN / 8), c = (q % (kBN / 8)) * 8;
      if (m0 + r < M && n0 + c < N)
        *reinterpret_cast<uint4*>(Y + size_t(m0 + r) * N + n0 + c) = *reinterpret_cast<const uint4*>(sX + size_t(r) * kOutStride + c * 2);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMMA) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_ex(const void* kern, dim3 grid, dim3 block, size_t smem, unsigned flags, cudaStream_t stream,
                      void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  int na = 0;
  if (flags & WQ_FLAG_PDL) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace

size_t w8a8_workspace_bytes(int M, int K, int N) {
  (void)N;
  if (M < 1 || K < 1) return 0;
  return align_up(size_t(M) * K * 2, 256) + align_up(size_t(M) * 4, 256);
}

// LLM.int8() needs, after the plain workspace, the column flags and the list
// of outlier columns (int [K] each), their count, and the gathered outlier
// activations (bf16 [K][M] at most: every column could be an outlier).
size_t w8a8_outlier_workspace_bytes(int M, int K, int N) {
  const size_t base = w8a8_workspace_bytes(M, K, N);
  if (base == 0) return 0;
  return base + 2 * align_up(size_t(K) * 4, 256) + 256 + align_up(size_t(K) * M * 2, 256);
}

cudaError_t launch_w8a8(const void* X, const int8_t* W, const float* Sw, void* Y, int M, int K, int N,
                        int8_t* Xq_out, float* Sx_out, int32_t* acc_out, void* workspace, unsigned flags,
                        cudaStream_t stream, const float* smooth, const float* outlier_threshold,
                        int32_t* n_outliers_out) {
  const SmemW8A8 L;
  if (L.total > static_cast<size_t>(device_max_smem())) return cudaErrorNotSupported;
  __half* xq16 = static_cast<__half*>(workspace);
  float* sx = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align_up(size_t(M) * K * 2, 256));
  const uint16_t* Xp = static_cast<const uint16_t*>(X);

  // 0) LLM.int8(): flag the outlier columns and list them
  int* oflags = nullptr;
  int* oidx = nullptr;
  int* ocount = nullptr;
  uint16_t* xoT = nullptr;
  if (outlier_threshold) {
    uint8_t* o = static_cast<uint8_t*>(workspace) + w8a8_workspace_bytes(M, K, N);
    oflags = reinterpret_cast<int*>(o);
    oidx = reinterpret_cast<int*>(o + align_up(size_t(K) * 4, 256));
    ocount = reinterpret_cast<int*>(o + 2 * align_up(size_t(K) * 4, 256));
    cudaError_t e = cudaMemsetAsync(oflags, 0, size_t(K) * 4, stream);
    if (e != cudaSuccess) return e;
    float th = *outlier_threshold;
    void* sargs[] = {&Xp, &M, &K, &th, &oflags};
    e = launch_ex(reinterpret_cast<const void*>(w8a8_outlier_scan_kernel),
                  dim3((K + 2047) / 2048, std::min((M + kScanRows - 1) / kScanRows, 65535)),
                  dim3(256), 0, flags, stream, sargs);
    if (e != cudaSuccess) return e;
    void* cargs[] = {&oflags, &K, &oidx, &ocount, &n_outliers_out};
    e = launch_ex(reinterpret_cast<const void*>(w8a8_outlier_compact_kernel), dim3(1), dim3(1024), 0,
                  flags | WQ_FLAG_PDL, stream, cargs);
    if (e != cudaSuccess) return e;
    xoT = reinterpret_cast<uint16_t*>(o + 2 * align_up(size_t(K) * 4, 256) + 256);
    void* gargs[] = {&Xp, &M, &K, &oidx, &ocount, &xoT};
    e = launch_ex(reinterpret_cast<const void*>(w8a8_outlier_gather_kernel), dim3((M + 255) / 256), dim3(256), 0,
                  flags | WQ_FLAG_PDL, stream, gargs);
    if (e != cudaSuccess) return e;
  }

  // 1) per-row quantization
  {
    const int* of = oflags;
    void* args[] = {&Xp, &K, &smooth, &of, &xq16, &sx, &Xq_out, &Sx_out};
    cudaError_t e = launch_ex(reinterpret_cast<const void*>(w8a8_quant_kernel), dim3(M), dim3(256), 0, flags, stream,
                              args);
    if (e != cudaSuccess) return e;
  }
  // 2) GEMM with the fused rescale epilogue (always chained to the quantization kernel)
  CUtensorMap xmap, wmap;
  if (!encode_tensor_map_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xq16, K, M, size_t(K) * 2, kBoxK, kBM,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, N, K, N, kBN, kBK, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  W8A8Args args{Sw, sx, Y, acc_out, oidx, ocount, xoT, outlier_threshold ? W : nullptr, M, K, N};
  const void* kern = outlier_threshold ? reinterpret_cast<const void*>(w8a8_mma_kernel<true>)
                                       : reinterpret_cast<const void*>(w8a8_mma_kernel<false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L.total));
  if (e != cudaSuccess) return e;
  void* kargs[] = {&xmap, &wmap, &args};
  return launch_ex(kern, dim3((N + kBN - 1) / kBN, (M + kBM - 1) / kBM), dim3(kThreads), L.total,
                   flags | WQ_FLAG_PDL, stream, kargs);
}

}  // namespace wq
