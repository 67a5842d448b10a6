// wq_gemv8.cu -- INT8 weight-only GEMV with group-wise fp32 scales.
//
// Definition ("Quantization CUDA", Int8 Weight Only Quantization: Y = (X.Wint)*Sw
// with fp32 accumulation; "融合反量化与GEMM", 量化策略：分组对称INT8: one fp32
// scale per group of 128 values of k):
//   y[m,n] = sum_k x[m,k] * s[k/group, n] * q[k,n].
// Storage: int8 [K, N], N contiguous.
//
// Exact conversion: XOR 0x80 turns the signed code into b = q + 128; PRMT puts
// b in the low byte of 0x4B000000 (= 2^23 + b exactly) and one packed FADD of
// -(2^23 + 128) returns q exactly.  The group scale multiplies the fp32 partial
// sum of each 8-row unit.
#include "wq_gemv_common.cuh"
#include "wq_launch.h"

namespace wq {
namespace {

constexpr int kBN = 256;           // int8 columns per tile: one 256-byte row per warp
constexpr int kUnitRows = 8;       // rows (= values of k) per consumer unit
constexpr int kStageRows = kConsumerWarps * kUnitRows;
constexpr int kStageBytes = kStageRows * kBN;  // 16 KB
constexpr int kNS = 4;

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

struct Smem8 {
  size_t xs, scl, part, bars, flag, total;
  __host__ __device__ Smem8(int MT, int ng_max) {
    size_t o = size_t(kNS) * kStageBytes;
    xs = o;   o = align16(o + size_t(kConsumerWarps) * MT * kUnitRows * 8);
    scl = o;  o = align16(o + size_t(ng_max) * kBN * 4);
    part = o; o = align16(o + size_t(MT) * kBN * 4);
    bars = o; o = align16(o + size_t(2 * kNS) * 8);
    flag = o; o = align16(o + 16);
    total = o;
  }
};

template <int MT>
__global__ void __launch_bounds__(kGemvThreads, 1)
    k8_gemv_kernel(const __grid_constant__ CUtensorMap wmap, const GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Smem8 L(MT, a.ng_max);
  uint8_t* stages = smem;
  float2* xs = reinterpret_cast<float2*>(smem + L.xs);
  float* scl = reinterpret_cast<float*>(smem + L.scl);
  float* part = reinterpret_cast<float*>(smem + L.part);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kNS;
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L.flag);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = gridDim.x, n0 = blockIdx.y * kBN;
  const int M = a.M, K = a.K, N = a.N, gsz = a.group;
  int u0, u1;
  split_range(K / kUnitRows, S, blockIdx.x, u0, u1);
  const int n_loads = (u1 - u0 + kConsumerWarps - 1) / kConsumerWarps;
  const int g0 = (kUnitRows * u0) / gsz;
  const int ng = (u1 > u0) ? (kUnitRows * u1 - 1) / gsz - g0 + 1 : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *failed = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    int issued = 0;
    if (lane == 0 && n_loads > 0)
      issued = produce_stages<kNS, kStageBytes>(&wmap, stages, full, empty, n0, kUnitRows * u0, kStageRows,
                                                n_loads, failed);
    pdl_wait();
    if (lane == 0 && *failed) drain_stages<kNS>(full, issued);
  } else {
    const float* X = static_cast<const float*>(a.x);
    const float* SC = static_cast<const float*>(a.scales);
    for (int i = threadIdx.x; i < ng * (kBN / 4); i += kConsumerThreads) {
      const int gr = i / (kBN / 4), c = 4 * (i % (kBN / 4));
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (n0 + c < N) v = *reinterpret_cast<const float4*>(SC + size_t(g0 + gr) * N + n0 + c);
      reinterpret_cast<float4*>(scl)[i] = v;
    }
    consumer_sync(kConsumerThreads);
    pdl_wait();

    float acc[MT][8];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[m][c] = 0.f;

    // x staging: the unit's 8 x MT values, lane l -> (m, j) = (l / 8 + 4 r, l % 8)
    constexpr int XR = (MT * kUnitRows + 31) / 32;
    float xnext[XR];
    auto load_x = [&](int u) {
#pragma unroll
      for (int r = 0; r < XR; ++r) {
        const int m = lane / kUnitRows + r * (32 / kUnitRows), j = lane % kUnitRows;
        xnext[r] = (u < u1 && m < M && m < MT) ? X[size_t(m) * K + kUnitRows * u + j] : 0.f;
      }
    };
    load_x(u0 + warp);
    float2* myxs = xs + warp * MT * kUnitRows;
    const float2 unbias = make_float2(-8388736.f, -8388736.f);  // -(2^23 + 128)

    for (int it = 0; it < n_loads; ++it) {
      const int s = it % kNS;
      const int u = u0 + it * kConsumerWarps + warp;
      const bool active = u < u1;
      __syncwarp();
#pragma unroll
      for (int r = 0; r < XR; ++r) {
        const int m = lane / kUnitRows + r * (32 / kUnitRows), j = lane % kUnitRows;
        if (m < MT) myxs[m * kUnitRows + j] = make_float2(xnext[r], xnext[r]);
      }
      __syncwarp();
      load_x(u + kConsumerWarps);
      if (!mbar_wait(&full[s], (it / kNS) & 1)) {
        *failed = 1;
        break;
      }
      if (active) {
        float2 accg[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int c = 0; c < 4; ++c) accg[m][c] = make_float2(0.f, 0.f);
        const uint8_t* rowp = stages + size_t(s) * kStageBytes + size_t(warp * kUnitRows) * kBN + lane * 8;
#pragma unroll
        for (int j = 0; j < kUnitRows; ++j) {
          const uint2 wd = *reinterpret_cast<const uint2*>(rowp + j * kBN);
          const uint32_t b0 = wd.x ^ 0x80808080u, b1 = wd.y ^ 0x80808080u;
          float2 q[4];
          q[0] = fadd2(make_float2(as_f32(prmt(b0, 0x4B000000u, 0x7440u)), as_f32(prmt(b0, 0x4B000000u, 0x7441u))), unbias);
          q[1] = fadd2(make_float2(as_f32(prmt(b0, 0x4B000000u, 0x7442u)), as_f32(prmt(b0, 0x4B000000u, 0x7443u))), unbias);
          q[2] = fadd2(make_float2(as_f32(prmt(b1, 0x4B000000u, 0x7440u)), as_f32(prmt(b1, 0x4B000000u, 0x7441u))), unbias);
          q[3] = fadd2(make_float2(as_f32(prmt(b1, 0x4B000000u, 0x7442u)), as_f32(prmt(b1, 0x4B000000u, 0x7443u))), unbias);
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const float2 xp = myxs[m * kUnitRows + j];
#pragma unroll
            for (int c = 0; c < 4; ++c) accg[m][c] = ffma2(xp, q[c], accg[m][c]);
          }
        }
        const int gi = (kUnitRows * u) / gsz - g0;
        const float4 sa = *reinterpret_cast<const float4*>(scl + gi * kBN + lane * 8);
        const float4 sb = *reinterpret_cast<const float4*>(scl + gi * kBN + lane * 8 + 4);
        const float s8[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            acc[m][2 * c] = fmaf(s8[2 * c], accg[m][c].x, acc[m][2 * c]);
            acc[m][2 * c + 1] = fmaf(s8[2 * c + 1], accg[m][c].y, acc[m][2 * c + 1]);
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    consumer_sync(kConsumerThreads);
    float* red = reinterpret_cast<float*>(stages);  // [8 warps][MT][BN] = 8 KB * MT <= 64 KB
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float* r = red + (warp * MT + m) * kBN + lane * 8;
      *reinterpret_cast<float4*>(r) = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
      *reinterpret_cast<float4*>(r + 4) = make_float4(acc[m][4], acc[m][5], acc[m][6], acc[m][7]);
    }
    consumer_sync(kConsumerThreads);
    for (int e = threadIdx.x; e < MT * kBN; e += kConsumerThreads) {
      const int m = e / kBN, col = e % kBN;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) v += red[(w * MT + m) * kBN + col];
      part[e] = v;
    }
  }

  float* Y = static_cast<float*>(a.y);
  finish_tile<MT, kBN>(part, S, [&](int m, int col, float v) {
    const int n = n0 + col;
    if (m < M && n < N) Y[size_t(m) * N + n] = v;
  });
}

}  // namespace

size_t wq8_gemv_smem_bytes(int MT, int ng_max) { return Smem8(MT, ng_max).total; }

cudaError_t launch_wq8_gemv(const LaunchPlan& p, const CUtensorMap& map, const GemvArgs& a) {
  const void* kern = nullptr;
  switch (p.MT) {
    case 1: kern = reinterpret_cast<const void*>(k8_gemv_kernel<1>); break;
    case 2: kern = reinterpret_cast<const void*>(k8_gemv_kernel<2>); break;
    case 4: kern = reinterpret_cast<const void*>(k8_gemv_kernel<4>); break;
    case 8: kern = reinterpret_cast<const void*>(k8_gemv_kernel<8>); break;
    default: return cudaErrorInvalidValue;
  }
  return launch_gemv_kernel(kern, p, Smem8(p.MT, a.ng_max).total, map, a);
}

}  // namespace wq
