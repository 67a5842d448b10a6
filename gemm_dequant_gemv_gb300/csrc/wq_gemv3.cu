// wq_gemv3.cu -- 3-bit GEMV with per-column fp16 scale and stored zero.
//
// Definition (GPTQ CUDA kernel walkthrough, CUDA核函數設計與實現):
//   y[m,n] = sum_k x[m,k] * (s[n] * q(k,n) - zero[n]),  zero[n] = s[n] * z[n] stored.
// Storage: int32 [3K/32, N]; the 32 codes of k = 32b..32b+31 of a column form
// a 96-bit little-endian bit stream over word rows 3b..3b+2, code j at bits
// [3j, 3j+3).
//
// Exact code conversion without extracting each code to bit 0: a word is
// shifted (or funnel-shifted across two words) so that four codes sit at bit
// offsets o in {11, 14, 17, 20}; AND with (7 << o) and OR with 0x3F000000 then
// gives the fp32 value m = 0.5 + q 2^(o-24) exactly.  The activation is staged
// pre-multiplied by 2^(24-o) (exact), so x' m = x 2^(23-o) + x q with an exact
// product; the per-CTA constant B = sum_k x_k 2^(23-o(k)) is removed once:
//   y = s (sum_k x' m - B) - zero * sum_k x.
#include "wq_gemv_common.cuh"
#include "wq_launch.h"

namespace wq {
namespace {

constexpr int kBN = 128;
constexpr int kUnitRows = 3;                       // one 32-code block
constexpr int kStageRows = kConsumerWarps * kUnitRows;
constexpr int kStageK = kConsumerWarps * 32;       // 256 values of k per stage
constexpr int kStageBytes = kStageRows * kBN * 4;  // 12 KB
constexpr int kNS = 5;

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

struct Smem3 {
  size_t xst, xc, recv, bars, flag, total;
  __host__ __device__ Smem3(int MT, int S) {
    size_t o = size_t(kNS) * kStageBytes;
    xst = o;  o = align16(o + size_t(kNS) * MT * kStageK * 2);
    xc = o;   o = align16(o + size_t(MT) * kStageK * 8);
    recv = o; o = align16(o + TileReduce(S, kBN).recv_floats(MT) * 4);
    bars = o; o = align16(o + size_t(2 * kNS + 1) * 8);
    flag = o; o = align16(o + 16);
    total = o;
  }
};

// Which of the nine shifted words holds code j of a block, and in which of its
// four slots (bit offset 11 + 3 * slot).  Shifts: w0<<11 (codes 0-3), w0>>1
// (4-7), w0>>13 (8-9), funnel(w0,w1)>>19 (10-13), w1<<1 (14-17),
// funnel(w1,w2)>>11 (18-21), w2<<9 (22-25), w2>>3 (26-29), w2>>15 (30-31).
__host__ __device__ constexpr int code_src(int j) {
  return j < 8 ? j / 4 : (j < 10 ? 2 : (j < 30 ? 3 + (j - 10) / 4 : 8));
}
__host__ __device__ constexpr int code_slot(int j) {
  return j < 8 ? j % 4 : (j < 10 ? j - 8 : (j < 30 ? (j - 10) % 4 : j - 30));
}
__host__ __device__ constexpr int code_offset(int j) { return 11 + 3 * code_slot(j); }

template <int MT>
__global__ void __launch_bounds__(kGemvThreads, 1)
    k3_gemv_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                   const GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Smem3 L(MT, gridDim.x);
  const TileReduce R(gridDim.x, kBN);
  uint8_t* wst = smem;
  uint8_t* xst = smem + L.xst;
  float2* xc = reinterpret_cast<float2*>(smem + L.xc);
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kNS;
  uint64_t* recv_bar = empty + kNS;
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L.flag);  // producer's
  volatile int* cfailed = failed + 1;                                       // consumers'

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = gridDim.x, n0 = blockIdx.y * kBN;
  const int M = a.M, K = a.K, N = a.N;
  int u0, u1;
  split_range(K / 32, S, blockIdx.x, u0, u1);
  const int n_loads = (u1 - u0 + kConsumerWarps - 1) / kConsumerWarps;
  constexpr uint32_t kXBytes = MT * kStageK * 2;

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
      issued = produce_stages<kNS>(&wmap, &xmap, wst, kStageBytes, xst, kXBytes, full, empty, n0, 3 * u0,
                                   kStageRows, 32 * u0, kStageK, n_loads, failed);
    pdl_wait();
    if (lane == 0 && *failed) drain_stages<kNS>(full, issued);
    __syncwarp();
    if (S > 1) cluster_wait();
  } else {
    const int tid = threadIdx.x;
    // this thread converts code position j = lane of every block it stages
    const int off = code_offset(lane);
    const float fac = __int_as_float((127 + 24 - off) << 23);   // 2^(24 - off)
    const float bfac = __int_as_float((127 + 23 - off) << 23);  // 2^(23 - off)
    float bsum[MT], xsum[MT];
    float2 acc[MT][2];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      bsum[m] = xsum[m] = 0.f;
      acc[m][0] = acc[m][1] = make_float2(0.f, 0.f);
    }
    // this lane's 4 columns' scale and stored zero: weight-side data, read before the dependency wait
    const __half* SC = static_cast<const __half*>(a.scales);
    const __half* ZR = static_cast<const __half*>(a.zeros);
    float sc[4], zr[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int n = n0 + 4 * lane + c;
      sc[c] = n < N ? __half2float(SC[n]) : 0.f;
      zr[c] = n < N ? __half2float(ZR[n]) : 0.f;
    }
    pdl_wait();
    const uint32_t magic = 0x3F000000u;

    float2* xcw = xc + warp * 32;
    for (int it = 0; it < n_loads; ++it) {
      const int s = it % kNS;
      const int u = u0 + it * kConsumerWarps + warp;
      if (!mbar_wait(&full[s], (it / kNS) & 1)) *cfailed = 1;
      if (*cfailed) break;
      {
        const __half* xr = reinterpret_cast<const __half*>(xst + size_t(s) * kXBytes) + warp * 32 + lane;
        const bool live = u < u1;  // k = 32u + lane belongs to this CTA's range
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const float v = live ? __half2float(xr[m * kStageK]) : 0.f;
          const float xp = v * fac;
          xcw[m * kStageK + lane] = make_float2(xp, xp);
          bsum[m] = fmaf(v, bfac, bsum[m]);
          xsum[m] += v;
        }
      }
      __syncwarp();
      if (u < u1) {
        const uint8_t* rowp = wst + size_t(s) * kStageBytes + size_t(warp * kUnitRows) * (kBN * 4) + lane * 16;
        const uint4 A = *reinterpret_cast<const uint4*>(rowp);
        const uint4 B = *reinterpret_cast<const uint4*>(rowp + kBN * 4);
        const uint4 C = *reinterpret_cast<const uint4*>(rowp + 2 * kBN * 4);
        const uint32_t w0[4] = {A.x, A.y, A.z, A.w};
        const uint32_t w1[4] = {B.x, B.y, B.z, B.w};
        const uint32_t w2[4] = {C.x, C.y, C.z, C.w};
        uint32_t t[4][9];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          t[c][0] = w0[c] << 11;
          t[c][1] = w0[c] >> 1;
          t[c][2] = w0[c] >> 13;
          t[c][3] = shf_r(w0[c], w1[c], 19);
          t[c][4] = w1[c] << 1;
          t[c][5] = shf_r(w1[c], w2[c], 11);
          t[c][6] = w2[c] << 9;
          t[c][7] = w2[c] >> 3;
          t[c][8] = w2[c] >> 15;
        }
        const float4* xw = reinterpret_cast<const float4*>(xcw);
#pragma unroll
        for (int jp = 0; jp < 16; ++jp) {
          float4 xq[MT];
#pragma unroll
          for (int m = 0; m < MT; ++m) xq[m] = xw[m * (kStageK / 2) + jp];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int j = 2 * jp + h;
            const uint32_t mask = 7u << code_offset(j);
            const int src = code_src(j);
            const float2 m01 = make_float2(as_f32(lop3_and_or(t[0][src], mask, magic)),
                                           as_f32(lop3_and_or(t[1][src], mask, magic)));
            const float2 m23 = make_float2(as_f32(lop3_and_or(t[2][src], mask, magic)),
                                           as_f32(lop3_and_or(t[3][src], mask, magic)));
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const float2 xp = h ? make_float2(xq[m].z, xq[m].w) : make_float2(xq[m].x, xq[m].y);
              acc[m][0] = ffma2(xp, m01, acc[m][0]);
              acc[m][1] = ffma2(xp, m23, acc[m][1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // this warp's share of y: s (sum x' m - B_w) - zero X_w over the k it handled
    // (B_w, X_w: butterfly sums over the lanes, the same value in every lane)
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float b = warp_sum(bsum[m]), x = warp_sum(xsum[m]);
      acc[m][0] = make_float2(fmaf(sc[0], acc[m][0].x - b, -zr[0] * x), fmaf(sc[1], acc[m][0].y - b, -zr[1] * x));
      acc[m][1] = make_float2(fmaf(sc[2], acc[m][1].x - b, -zr[2] * x), fmaf(sc[3], acc[m][1].y - b, -zr[3] * x));
    }
    push_partials<MT, kBN>(R, acc, recv, recv_bar, warp, lane);
  }

  __half* Y = static_cast<__half*>(a.y);
  owner_reduce_store<MT, kBN>(R, recv, recv_bar, [&](int m, int col, float v) {
    const int n = n0 + col;
    if (m < M && n < N) Y[size_t(m) * N + n] = __float2half_rn(v);
  });
}

}  // namespace

size_t wq3_gemv_smem_bytes(int MT, int S) { return Smem3(MT, S).total; }

int wq3_stage_k() { return kStageK; }

cudaError_t launch_wq3_gemv(const LaunchPlan& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                            const GemvArgs& a) {
  const void* kern = nullptr;
  switch (p.MT) {
    case 1: kern = reinterpret_cast<const void*>(k3_gemv_kernel<1>); break;
    case 2: kern = reinterpret_cast<const void*>(k3_gemv_kernel<2>); break;
    case 4: kern = reinterpret_cast<const void*>(k3_gemv_kernel<4>); break;
    case 8: kern = reinterpret_cast<const void*>(k3_gemv_kernel<8>); break;
    default: return cudaErrorInvalidValue;
  }
  const CUtensorMap* maps[2] = {&wmap, &xmap};
  return launch_gemv_kernel(kern, p, Smem3(p.MT, p.S).total, maps, 2, a);
}

}  // namespace wq
