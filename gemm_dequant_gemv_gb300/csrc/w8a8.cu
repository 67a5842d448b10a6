// w8a8.cu -- W8A8 dynamic-quantization GEMM on the tcgen05 tensor cores.
//
// Definition ("Quantization CUDA", Dynamic Quantization and 优化):
//   Sx[m]    = fp32(max_k |X[m,k]| / 127)          (activations quantized at run time, per token)
//   Xq[m,k]  = clamp(rint(fp32(X[m,k] / Sx[m])), -127, 127)
//   acc[m,n] = sum_k Xq[m,k] * W[k,n]              (int8 multiply, exact int32 accumulate)
//   Y[m,n]   = bf16(Sx[m] * acc[m,n] * Sw[n])      (rescale fused into the matmul epilogue)
//
// sm_103a has no integer tcgen05 MMA, so the product runs as kind::f16 on
// fp16 operands that hold the integer codes exactly (|q| <= 127).  Every
// product is an exact integer and so is every partial sum below 2^24: the
// tensor core accumulates 256 values of k (|sum| <= 256 * 127^2 < 2^22) into
// an fp32 tensor-memory accumulator, and the epilogue warps fold each such
// chunk into an int32 register sum with the magic-number conversion
// bits(f + 1.5 * 2^23) (exact for |f| < 2^22; the constant is removed once at
// the end, in wrapping unsigned arithmetic).  The int32 result is never
// stored unless a debug output is requested.
//
// Kernels: (1) w8a8_quant_kernel, one CTA per row: Sx, the int8 codes (if
// requested) and fp16 copies of the codes in the workspace; (2)
// w8a8_mma_kernel, one 128 x 128 output tile per CTA:
//   warp 8 : TMA of the fp16 code tile of X (128-byte swizzle) and the int8
//            tile of W [64 k x 128 n] per 64-value k-stage;
//   warps 0-3 : convert the int8 W tile to fp16 (exact) in the MN-major
//            128-byte-swizzled layout of the B operand;
//   warp 9 : four MMAs (M = N = 128, K = 16) per stage into one of two
//            tensor-memory accumulators (one per 256-value chunk);
//   warps 4-7 : drain each chunk into int32 and, at the end, write
//            Y = bf16(Sx * acc * Sw) through shared memory with coalesced stores.
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
__global__ void __launch_bounds__(256) w8a8_quant_kernel(const uint16_t* __restrict__ X, int K,
                                                         __half* __restrict__ xq16, float* __restrict__ sx_ws,
                                                         int8_t* __restrict__ xq_out, float* __restrict__ sx_out) {
  __shared__ float red[8];
  const int m = blockIdx.x;
  pdl_wait();
  const uint16_t* row = X + size_t(m) * K;
  float amax = 0.f;
  for (int k = threadIdx.x * 8; k < K; k += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w[i] & 0xFFFFu)));
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w[i] >> 16)));
    }
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
    const uint4 v = *reinterpret_cast<const uint4*>(row + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    int q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float x = bf16_bits_to_f32((i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu));
      int c = 0;
      if (sx != 0.f) c = min(127, max(-127, __float2int_rn(__fdiv_rn(x, sx))));
      q[i] = c;
    }
    uint4 h;
    h.x = uint32_t(__half_as_ushort(__int2half_rn(q[0]))) | (uint32_t(__half_as_ushort(__int2half_rn(q[1]))) << 16);
    h.y = uint32_t(__half_as_ushort(__int2half_rn(q[2]))) | (uint32_t(__half_as_ushort(__int2half_rn(q[3]))) << 16);
    h.z = uint32_t(__half_as_ushort(__int2half_rn(q[4]))) | (uint32_t(__half_as_ushort(__int2half_rn(q[5]))) << 16);
    h.w = uint32_t(__half_as_ushort(__int2half_rn(q[6]))) | (uint32_t(__half_as_ushort(__int2half_rn(q[7]))) << 16);
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

// --------------------------------------------------------------------- GEMM --
constexpr int kBM = 128, kBN = 128, kBK = 128;
constexpr int kBoxK = 64;                    // values of k per 128-byte-swizzled X box
constexpr int kChunkStages = 256 / kBK;      // 256 values of k per exact fp32 chunk
constexpr int kNS = 3, kNB = 2;
constexpr int kConvWarps = 8;            // int8 -> fp16 converters of the B tile
constexpr int kEpiWarps = 8;             // two per tensor-memory lane quarter, 64 columns each
constexpr int kThreads = (kConvWarps + kEpiWarps + 2) * 32;
constexpr int kWarpTMA = kConvWarps + kEpiWarps, kWarpMMA = kWarpTMA + 1;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kEpiCols = kBN / (kEpiWarps / 4);  // columns per epilogue thread
constexpr int kABoxBytes = kBM * kBoxK * 2;  // 16 KB: one X box (128 rows x 64 k)
constexpr int kABytes = kBM * kBK * 2;       // 32 KB fp16 codes of X per stage (two boxes)
constexpr int kWBytes = kBK * kBN;           // 16 KB int8 W
constexpr int kBBytes = kBN * kBK * 2;       // 32 KB fp16 W in the MN-major layout
// MN-major 128-byte-swizzle atoms of the B operand: 8 rows of k x 64 values of n.
constexpr uint32_t kAtomK = 1024;                      // byte stride between k-atoms (adjacent)
constexpr uint32_t kAtomN = (kBK / 8) * kAtomK;        // byte stride between the two n-atoms
constexpr int kOutStride = kBN * 2 + 16; // padded bf16 output row in shared memory

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) & ~(a - 1); }

struct SmemW8A8 {
  size_t a, w, b, sw, sx, bars, misc, total;
  __host__ __device__ SmemW8A8() {
    size_t o = 0;
    a = o;    o += size_t(kNS) * kABytes;     // also the output staging area at the end
    b = o;    o += size_t(kNB) * kBBytes;
    w = o;    o += size_t(kNS) * kWBytes;
    sw = o;   o = align_up(o + kBN * 4, 16);
    sx = o;   o = align_up(o + kBM * 4, 16);
    bars = o; o = align_up(o + size_t(4 * kNS + 2 * kNB + 4) * 8, 16);
    misc = o; o = align_up(o + 32, 16);
    total = o + 1024;
  }
};

// MN-major, 128-byte-swizzle descriptor: leading-dimension offset = stride
// between the 64-wide n-atoms, stride-dimension offset = stride between the
// 8-row k-atoms.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((kAtomN >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((kAtomK >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

struct W8A8Args {
  const float* Sw;
  const float* Sx;       // workspace copy written by the quantization kernel
  void* Y;               // bf16 [M, N]
  int32_t* acc_out;      // optional
  int M, K, N;
};

__global__ void __launch_bounds__(kThreads, 1)
    w8a8_mma_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap wmap,
                    const W8A8Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemW8A8 L;
  uint8_t* sA = smem + L.a;
  uint8_t* sB = smem + L.b;
  uint8_t* sW = smem + L.w;
  float* sSw = reinterpret_cast<float*>(smem + L.sw);
  float* sSx = reinterpret_cast<float*>(smem + L.sx);
  // full / empty: the X-code ring (released when the MMA has read a stage);
  // wfull / wempty: the int8 W ring (released as soon as the converters have read it)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kNS;
  uint64_t* wfull = empty + kNS;
  uint64_t* wempty = wfull + kNS;
  uint64_t* b_full = wempty + kNS;
  uint64_t* b_empty = b_full + kNB;
  uint64_t* t_full = b_empty + kNB;
  uint64_t* t_empty = t_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L.misc + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM;
  const int M = a.M, K = a.K, N = a.N;
  const int nst = (K + kBK - 1) / kBK;  // the tail of the last stage is zero-filled by TMA
  const int nchunks = (nst + kChunkStages - 1) / kChunkStages;
  constexpr uint32_t kTmemCols = 2 * kBN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], kConvWarps * 32);
    }
    for (int s = 0; s < kNB; ++s) {
      mbar_init(&b_full[s], kConvWarps * 32);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&t_full[s], 1);
      mbar_init(&t_empty[s], kEpiThreads);
    }
    *failed = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  if (warp == kWarpTMA) {
    // ------------------------------------------------------------ producer --
    // lane 0 streams the int8 W tiles (weight-side data: no dependency wait, the
    // converters can start before the previous kernel has finished); lane 1
    // streams the fp16 X codes after the wait.
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      for (int i = 0; i < nst && !*failed; ++i) {
        const int s = i % kNS;
        if (i >= kNS && !mbar_wait(&wempty[s], ((i / kNS) - 1) & 1)) {
          *failed = 1;
          break;
        }
        mbar_expect_tx(&wfull[s], kWBytes);
        tma_load_2d(sW + size_t(s) * kWBytes, &wmap, &wfull[s], n0, i * kBK, 0ull);
      }
    } else if (lane == 1) {
      prefetch_tensormap(&amap);
      pdl_wait();
      for (int i = 0; i < nst && !*failed; ++i) {
        const int s = i % kNS;
        if (i >= kNS && !mbar_wait(&empty[s], ((i / kNS) - 1) & 1)) {
          *failed = 1;
          break;
        }
        mbar_expect_tx(&full[s], kABytes);
#pragma unroll
        for (int h = 0; h < kBK / kBoxK; ++h)
          tma_load_2d(sA + size_t(s) * kABytes + h * kABoxBytes, &amap, &full[s], i * kBK + h * kBoxK, m0, 0ull);
      }
    } else {
      pdl_wait();
    }
  } else if (warp == kWarpMMA) {
    // ----------------------------------------------------------------- MMA --
    pdl_wait();
    if (lane == 0) {
      // fp32 accumulator, fp16 A (K-major) and B (MN-major), M = N = 128
      const uint32_t idesc = (1u << 4) | (1u << 16) | (uint32_t(kBN >> 3) << 17) | (uint32_t(kBM >> 4) << 24);
      int last = -1;
      for (int i = 0; i < nst; ++i) {
        const int s = i % kNS, bb = i % kNB, ch = i / kChunkStages, tb = ch & 1;
        if (i % kChunkStages == 0 && ch >= 2) {
          if (!mbar_wait(&t_empty[tb], ((ch / 2) - 1) & 1)) { *failed = 1; break; }
        }
        if (!mbar_wait(&b_full[bb], (i / kNB) & 1) || !mbar_wait(&full[s], (i / kNS) & 1)) {
          *failed = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(sA + size_t(s) * kABytes);
        const uint32_t b_base = smem_u32(sB + size_t(bb) * kBBytes);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_f16(tmem + tb * kBN, sw128_kmajor_desc(a_base + (k / (kBoxK / 16)) * kABoxBytes + 32 * (k % (kBoxK / 16))),
                  sw128_mnmajor_desc(b_base + 2 * kAtomK * k),
                  idesc, (i % kChunkStages != 0 || k > 0) ? 1u : 0u);
        mma_commit(&empty[s]);
        mma_commit(&b_empty[bb]);
        if (i % kChunkStages == kChunkStages - 1 || i == nst - 1) mma_commit(&t_full[tb]);
        last = i;
      }
      if (last >= 0) mbar_wait(&empty[last % kNS], (last / kNS) & 1);
    }
  } else if (warp < kConvWarps) {
    // ---------------------------------------------------------- converters --
    const int t = threadIdx.x;  // 0 .. kConvWarps * 32 - 1
    for (int i = 0; i < nst; ++i) {
      const int s = i % kNS, bb = i % kNB;
      if (!mbar_wait(&wfull[s], (i / kNS) & 1)) { *failed = 1; break; }
      if (i >= kNB && !mbar_wait(&b_empty[bb], ((i / kNB) - 1) & 1)) { *failed = 1; break; }
      const uint8_t* wt = sW + size_t(s) * kWBytes;
      uint8_t* bt = sB + size_t(bb) * kBBytes;
#pragma unroll
      for (int p = 0; p < (kWBytes / 16) / (kConvWarps * 32); ++p) {
        // 16-byte chunk (row k, columns 16c..16c+15) of the int8 tile.  Within each
        // 8-lane phase k % 8 = i runs over 0..7 and c = (i + d) % 8, so that the
        // loads (chunk c of a 128-byte row) and both swizzled stores (chunk
        // (2 (c % 4) [+1]) ^ (k % 8)) hit 8 different bank groups.
        const int q = t + kConvWarps * 32 * p;
        const int i = q & 7, rest = q >> 3;
        const int k = 8 * (rest % (kBK / 8)) + i, c = (i + rest / (kBK / 8)) & 7;
        const uint4 v = *reinterpret_cast<const uint4*>(wt + k * kBN + c * 16);
        const uint32_t w4[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
        uint32_t h[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // bytes b = q + 128 -> fp16 1024 + b, minus 1152 -> q exactly
          h[2 * j] = prmt(w4[j], 0x64646464u, 0x4140u);
          h[2 * j + 1] = prmt(w4[j], 0x64646464u, 0x4342u);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t d;
          asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(h[j]), "r"(0x64806480u));
          h[j] = d;
        }
        const int ka = k >> 3, r = k & 7, na = c >> 2, cc = 2 * (c & 3);
        uint8_t* rowp = bt + ka * kAtomK + na * kAtomN + r * 128;
        *reinterpret_cast<uint4*>(rowp + ((cc ^ r) * 16)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(rowp + (((cc + 1) ^ r) * 16)) = make_uint4(h[4], h[5], h[6], h[7]);
      }
      mbar_arrive(&wempty[s]);  // this thread's reads of the W stage are done (values in registers)
      fence_async_smem();
      mbar_arrive(&b_full[bb]);
    }
    pdl_wait();
  } else {
    // ------------------------------------------------------------ epilogue --
    // warp e (0..7): tensor-memory lane quarter e % 4 = tile rows 32 (e % 4) ..,
    // columns kEpiCols * (e / 4) ..
    pdl_wait();
    const int et = threadIdx.x - kConvWarps * 32;  // 0 .. kEpiThreads - 1
    const int ew = warp - kConvWarps, quarter = ew & 3, half = ew >> 2;
    const int row = quarter * 32 + lane;            // tensor-memory lane == output row in the tile
    const int cbase = half * kEpiCols;
    for (int c = et; c < kBN; c += kEpiThreads) sSw[c] = (n0 + c < N) ? a.Sw[n0 + c] : 0.f;
    if (half == 0) sSx[row] = (m0 + row < M) ? a.Sx[m0 + row] : 0.f;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + cbase;
    uint32_t acc[kEpiCols];
#pragma unroll
    for (int c = 0; c < kEpiCols; ++c) acc[c] = 0u;
    int drained = 0;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int tb = ch & 1;
      if (!mbar_wait(&t_full[tb], (ch / 2) & 1)) { *failed = 1; break; }
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < kEpiCols; c0 += 16) {
        float v[16];
        tmem_ld16(lane_addr + tb * kBN + c0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[c0 + j] += __float_as_uint(v[j] + 12582912.0f);
      }
      tc_fence_before();
      mbar_arrive(&t_empty[tb]);
      ++drained;
    }
    const uint32_t bias = uint32_t(drained) * 0x4B400000u;
    // Y = bf16(Sx * acc * Sw) staged in shared memory (the X stages are free now)
    asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");  // epilogue warps: sSw / sSx complete
    const float sx = sSx[row];
    uint8_t* orow = sA + size_t(row) * kOutStride + cbase * 2;
#pragma unroll
    for (int c0 = 0; c0 < kEpiCols; c0 += 8) {
      uint32_t pk[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int32_t i0 = static_cast<int32_t>(acc[c0 + 2 * j] - bias);
        const int32_t i1 = static_cast<int32_t>(acc[c0 + 2 * j + 1] - bias);
        const float f0 = (sx * static_cast<float>(i0)) * sSw[cbase + c0 + 2 * j];
        const float f1 = (sx * static_cast<float>(i1)) * sSw[cbase + c0 + 2 * j + 1];
        pk[j] = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(f0))) |
                (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(f1))) << 16);
      }
      *reinterpret_cast<uint4*>(orow + c0 * 2) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      if (a.acc_out && m0 + row < M) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (n0 + cbase + c0 + j < N)
            a.acc_out[size_t(m0 + row) * N + n0 + cbase + c0 + j] = static_cast<int32_t>(acc[c0 + j] - bias);
      }
    }
    asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");
    // coalesced stores: 16 chunks of 16 bytes per tile row
    uint16_t* Y = static_cast<uint16_t*>(a.Y);
    for (int q = et; q < kBM * (kBN / 8); q += kEpiThreads) {
      const int r = q / (kBN / 8), c = (q % (kBN / 8)) * 8;
      if (m0 + r < M && n0 + c < N)
        *reinterpret_cast<uint4*>(Y + size_t(m0 + r) * N + n0 + c) = *reinterpret_cast<const uint4*>(sA + size_t(r) * kOutStride + c * 2);
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

cudaError_t launch_w8a8(const void* X, const int8_t* W, const float* Sw, void* Y, int M, int K, int N,
                        int8_t* Xq_out, float* Sx_out, int32_t* acc_out, void* workspace, unsigned flags,
                        cudaStream_t stream) {
  const SmemW8A8 L;
  if (L.total > static_cast<size_t>(device_max_smem())) return cudaErrorNotSupported;
  __half* xq16 = static_cast<__half*>(workspace);
  float* sx = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align_up(size_t(M) * K * 2, 256));

  // 1) per-row quantization
  {
    const uint16_t* Xp = static_cast<const uint16_t*>(X);
    void* args[] = {&Xp, &K, &xq16, &sx, &Xq_out, &Sx_out};
    cudaError_t e = launch_ex(reinterpret_cast<const void*>(w8a8_quant_kernel), dim3(M), dim3(256), 0, flags, stream,
                              args);
    if (e != cudaSuccess) return e;
  }
  // 2) GEMM with the fused rescale epilogue (always chained to the quantization kernel)
  CUtensorMap amap, wmap;
  if (!encode_tensor_map_2d(&amap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xq16, K, M, size_t(K) * 2, kBoxK, kBM,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, N, K, N, kBN, kBK, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  W8A8Args args{Sw, sx, Y, acc_out, M, K, N};
  const void* kern = reinterpret_cast<const void*>(w8a8_mma_kernel);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L.total));
  if (e != cudaSuccess) return e;
  void* kargs[] = {&amap, &wmap, &args};
  return launch_ex(kern, dim3((N + kBN - 1) / kBN, (M + kBM - 1) / kBM), dim3(kThreads), L.total,
                   flags | WQ_FLAG_PDL, stream, kargs);
}

}  // namespace wq
