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
// sum of each 8-row unit.  One warp row is 128 int8 columns (4 per thread).
#include "wq_gemv_common.cuh"
#include "wq_launch.h"

namespace wq {
namespace {

constexpr int kBN = 128;           // int8 columns per tile: one 128-byte row per warp
constexpr int kUnitRows = 16;      // rows (= values of k) per consumer unit
constexpr int kStageRows = kConsumerWarps * kUnitRows;
constexpr int kStageK = kStageRows;            // 128 values of k per stage
constexpr int kStageBytes = kStageRows * kBN;  // 16 KB
constexpr int kNS = 4;

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

struct Smem8 {
  size_t xst, xc, scl, recv, bars, flag, total;
  __host__ __device__ Smem8(int MT, int ng_max, int S) {
    size_t o = size_t(kNS) * kStageBytes;
    xst = o;  o = align16(o + size_t(kNS) * MT * kStageK * 4);
    xc = o;   o = align16(o + size_t(MT) * kStageK * 8);
    scl = o;  o = align16(o + size_t(ng_max) * kBN * 4);
    recv = o; o = align16(o + TileReduce(S, kBN).recv_floats(MT) * 4);
    bars = o; o = align16(o + size_t(2 * kNS + 1) * 8);
    flag = o; o = align16(o + 16);
    total = o;
  }
};

template <int MT>
__global__ void __launch_bounds__(kGemvThreads, 1)
    k8_gemv_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                   const GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Smem8 L(MT, a.ng_max, gridDim.x);
  const TileReduce R(gridDim.x, kBN);
  uint8_t* wst = smem;
  uint8_t* xst = smem + L.xst;
  float2* xc = reinterpret_cast<float2*>(smem + L.xc);
  float* scl = reinterpret_cast<float*>(smem + L.scl);
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kNS;
  uint64_t* recv_bar = empty + kNS;
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L.flag);  // producer's
  volatile int* cfailed = failed + 1;                                       // consumers'

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = gridDim.x, n0 = blockIdx.y * kBN;
  const int M = a.M, K = a.K, N = a.N, gsz = a.group;
  int u0, u1;
  split_range(K / kUnitRows, S, blockIdx.x, u0, u1);
  const int n_loads = (u1 - u0 + kConsumerWarps - 1) / kConsumerWarps;
  const UnitGroups ug(gsz, kUnitRows);
  const int g0 = ug.of(u0);
  const int ng = (u1 > u0) ? (kUnitRows * u1 - 1) / gsz - g0 + 1 : 0;
  constexpr uint32_t kXBytes = MT * kStageK * 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *failed = 0;
    *cfailed = 0;
    R.init_bar(recv_bar, MT, kBN);
    fence_mbar_init();
  }
  __syncthreads();
  if (S > 1) cluster_arrive_relaxed();
  pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    int issued = 0;
    if (lane == 0 && n_loads > 0)
      issued = produce_stages<kNS>(&wmap, &xmap, wst, kStageBytes, xst, kXBytes, full, empty, n0, kUnitRows * u0,
                                   kStageRows, kUnitRows * u0, kStageK, n_loads, failed);
    pdl_wait();
    if (lane == 0 && *failed) drain_stages<kNS>(full, issued);
    __syncwarp();
    if (S > 1) cluster_wait();
  } else {
    const int tid = threadIdx.x;
    // the CTA's scale rows: weight-side data, requested before the dependency
    // wait but stored after it -- a store right after its load would hold the
    // thread (and its wait) for the whole HBM latency; the first two float4 of
    // each thread (all of them up to 16 groups) stay in registers meanwhile
    const float* SC = static_cast<const float*>(a.scales);
    const int nsc = ng * (kBN / 4);
    auto scale4 = [&](int i) {
      const int gr = i / (kBN / 4), c = 4 * (i % (kBN / 4));
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < nsc && n0 + c < N) v = *reinterpret_cast<const float4*>(SC + size_t(g0 + gr) * N + n0 + c);
      return v;
    };
    const float4 s0 = scale4(tid), s1 = scale4(tid + kConsumerThreads);
    pdl_wait();
    if (tid < nsc) reinterpret_cast<float4*>(scl)[tid] = s0;
    if (tid + kConsumerThreads < nsc) reinterpret_cast<float4*>(scl)[tid + kConsumerThreads] = s1;
    for (int i = tid + 2 * kConsumerThreads; i < nsc; i += kConsumerThreads) reinterpret_cast<float4*>(scl)[i] = scale4(i);
    consumer_sync(kConsumerThreads);  // the scale table is complete before any warp folds

    float2 acc[MT][2];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = make_float2(0.f, 0.f);
    const float2 unbias = make_float2(-8388736.f, -8388736.f);  // -(2^23 + 128)

    float2* xcw = xc + warp * kUnitRows;
    for (int it = 0; it < n_loads; ++it) {
      const int s = it % kNS;
      const int u = u0 + it * kConsumerWarps + warp;
      if (!mbar_wait(&full[s], (it / kNS) & 1)) *cfailed = 1;
      if (*cfailed) break;
      {
        // this warp's 16 values of x for every row: lane -> (m, j) = (lane / 16 + 2 r, lane % 16)
        const float* xr = reinterpret_cast<const float*>(xst + size_t(s) * kXBytes) + warp * kUnitRows;
#pragma unroll
        for (int r = 0; r < (MT * kUnitRows + 31) / 32; ++r) {
          const int m = lane / kUnitRows + r * (32 / kUnitRows), j = lane % kUnitRows;
          if (m < MT) {
            const float v = xr[m * kStageK + j];
            xcw[m * kStageK + j] = make_float2(v, v);
          }
        }
      }
      __syncwarp();
      if (u < u1) {
        float2 accg[MT][2];
#pragma unroll
        for (int m = 0; m < MT; ++m) accg[m][0] = accg[m][1] = make_float2(0.f, 0.f);
        const uint8_t* rowp = wst + size_t(s) * kStageBytes + size_t(warp * kUnitRows) * kBN + lane * 4;
        const float4* xw = reinterpret_cast<const float4*>(xcw);
#pragma unroll
        for (int jp = 0; jp < kUnitRows / 2; ++jp) {
          float4 xq[MT];
#pragma unroll
          for (int m = 0; m < MT; ++m) xq[m] = xw[m * (kStageK / 2) + jp];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t b = *reinterpret_cast<const uint32_t*>(rowp + (2 * jp + h) * kBN) ^ 0x80808080u;
            const float2 q01 = fadd2(make_float2(as_f32(prmt(b, 0x4B000000u, 0x7440u)), as_f32(prmt(b, 0x4B000000u, 0x7441u))), unbias);
            const float2 q23 = fadd2(make_float2(as_f32(prmt(b, 0x4B000000u, 0x7442u)), as_f32(prmt(b, 0x4B000000u, 0x7443u))), unbias);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const float2 xp = h ? make_float2(xq[m].z, xq[m].w) : make_float2(xq[m].x, xq[m].y);
              accg[m][0] = ffma2(xp, q01, accg[m][0]);
              accg[m][1] = ffma2(xp, q23, accg[m][1]);
            }
          }
        }
        const int gi = ug.of(u) - g0;
        const float4 sv = *reinterpret_cast<const float4*>(scl + gi * kBN + lane * 4);
        const float2 s01 = make_float2(sv.x, sv.y), s23 = make_float2(sv.z, sv.w);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          acc[m][0] = ffma2(s01, accg[m][0], acc[m][0]);
          acc[m][1] = ffma2(s23, accg[m][1], acc[m][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    push_partials<MT, kBN>(R, acc, recv, recv_bar, warp, lane);
  }

  float* Y = static_cast<float*>(a.y);
  owner_reduce_store<MT, kBN>(R, recv, recv_bar, [&](int m, int col, float v) {
    const int n = n0 + col;
    if (m < M && n < N) Y[size_t(m) * N + n] = v;
  });
}

}  // namespace

size_t wq8_gemv_smem_bytes(int MT, int ng_max, int S) { return Smem8(MT, ng_max, S).total; }

int wq8_stage_k() { return kStageK; }

cudaError_t launch_wq8_gemv(const LaunchPlan& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                            const GemvArgs& a) {
  const void* kern = nullptr;
  switch (p.MT) {
    case 1: kern = reinterpret_cast<const void*>(k8_gemv_kernel<1>); break;
    case 2: kern = reinterpret_cast<const void*>(k8_gemv_kernel<2>); break;
    case 4: kern = reinterpret_cast<const void*>(k8_gemv_kernel<4>); break;
    case 8: kern = reinterpret_cast<const void*>(k8_gemv_kernel<8>); break;
    default: return cudaErrorInvalidValue;
  }
  const CUtensorMap* maps[2] = {&wmap, &xmap};
  return launch_gemv_kernel(kern, p, Smem8(p.MT, a.ng_max, p.S).total, maps, 2, a);
}

}  // namespace wq
