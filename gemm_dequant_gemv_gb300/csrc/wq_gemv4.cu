// wq_gemv4.cu -- 4-bit group-wise weight-only GEMV / skinny GEMM on CUDA cores
// (M <= 8), with and without act-order.
//
// Definition ("Quantization CUDA", Weight Only Quantization / 量化粒度 and
// Marlin 格式):  y[m,n] = sum_k x[m,k] * s[g(k),n] * (q(k,n) - z[g(k),n]).
// Storage: qweight int32 [K/8, N], nibble j of word [r, n] = code of row 8r+j
// ("Int4 Weight Only Quantization / Weight Store": codes consecutive along K).
//
// Exact code conversion.  PRMT places a nibble q (0..15, high nibble already
// cleared) in byte 2 of the word 0x3F000000, which is the fp32 value
// m = 0.5 + q/256 exactly.  With x' = 256 x (exact), x' * m = 128 x + x q is
// an exact product (at most 19 significant bits), so the only rounding is the
// fp32 accumulation.  The constant 128 x is removed per group at the end:
//   contiguous groups:  y = sum_g s_g * (sum_{k in g} x' m_k - (128 + z_g) X_g)
//   act-order        :  w = fma(s, m, d) with d = -s (0.5 + z/256) is exactly
//                       s (q - z) / 256, and acc += x' w.
#include "wq_gemv_common.cuh"
#include "wq_launch.h"

namespace wq {
namespace {

constexpr int kBN = 128;          // columns per tile (one 512-byte row per warp)
constexpr int kUnitRows = 4;      // packed rows per consumer unit (32 values of k)
constexpr int kStageRows = kConsumerWarps * kUnitRows;
constexpr int kStageBytes = kStageRows * kBN * 4;  // 16 KB
constexpr int kNS = 4;

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

// Shared-memory carve-up (same arithmetic on host and device).
struct Smem4 {
  size_t xs, aux, zw, xg, part, bars, flag, total;
  __host__ __device__ Smem4(int MT, int ng_max, bool act_order, int G) {
    size_t o = size_t(kNS) * kStageBytes;
    xs = o;   o = align16(o + size_t(kConsumerWarps) * MT * 32 * 8);
    aux = o;  // contiguous: raw 16-bit scales [ng_max][BN]; act-order: per-warp goff [8][32] + sd [G][BN] float2
    if (act_order) o = align16(o + size_t(kConsumerWarps) * 32 * 4 + size_t(G) * kBN * 8);
    else           o = align16(o + size_t(ng_max) * kBN * 2);
    zw = o;   o = align16(o + (act_order ? 0 : size_t(ng_max) * (kBN / 8) * 4));
    xg = o;   o = align16(o + (act_order ? 0 : size_t(MT) * ng_max * 4));
    part = o; o = align16(o + size_t(MT) * kBN * 4);
    bars = o; o = align16(o + size_t(2 * kNS) * 8);
    flag = o; o = align16(o + 16);
    total = o;
  }
};

template <int ACT_BF16>
__device__ __forceinline__ float scale_bits_to_f32(uint32_t bits16) {
  return ACT_BF16 ? bf16_bits_to_f32(bits16) : f16_bits_to_f32(bits16);
}

// ---------------------------------------------------------------------------
// Contiguous groups (g(k) = k / group).
// ---------------------------------------------------------------------------
template <int MT, int ACT_BF16, bool HAS_Z>
__global__ void __launch_bounds__(kGemvThreads, 1)
    k4_gemv_kernel(const __grid_constant__ CUtensorMap wmap, const GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Smem4 L(MT, a.ng_max, false, 0);
  uint8_t* stages = smem;
  float2* xs = reinterpret_cast<float2*>(smem + L.xs);
  uint16_t* scl = reinterpret_cast<uint16_t*>(smem + L.aux);
  uint32_t* zw = reinterpret_cast<uint32_t*>(smem + L.zw);
  float* xg = reinterpret_cast<float*>(smem + L.xg);
  float* part = reinterpret_cast<float*>(smem + L.part);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kNS;
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L.flag);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = gridDim.x, n0 = blockIdx.y * kBN;
  const int M = a.M, K = a.K, N = a.N, gsz = a.group;
  int u0, u1;
  split_range(K / 32, S, blockIdx.x, u0, u1);
  const int n_loads = (u1 - u0 + kConsumerWarps - 1) / kConsumerWarps;
  const int g0 = (32 * u0) / gsz;
  const int ng = (u1 > u0) ? (32 * u1 - 1) / gsz - g0 + 1 : 0;

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

  float acc[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[m][c] = 0.f;

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    int issued = 0;
    if (lane == 0 && n_loads > 0)
      issued = produce_stages<kNS, kStageBytes>(&wmap, stages, full, empty, n0, 4 * u0, kStageRows, n_loads,
                                                failed);
    pdl_wait();
    if (lane == 0 && *failed) drain_stages<kNS>(full, issued);
  } else {
    // ---------------- consumers ----------------
    const uint16_t* X = static_cast<const uint16_t*>(a.x);
    // scale (and zero) slice of this CTA: weight-side data, read before the dependency wait
    for (int i = threadIdx.x; i < ng * (kBN / 2); i += kConsumerThreads) {
      const int gr = i / (kBN / 2), c = 2 * (i % (kBN / 2));
      uint32_t v = 0;
      if (n0 + c < N)
        v = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(a.scales) +
                                               size_t(g0 + gr) * N + n0 + c);
      reinterpret_cast<uint32_t*>(scl)[i] = v;
    }
    if (HAS_Z) {
      const int32_t* qz = static_cast<const int32_t*>(a.zeros);
      for (int i = threadIdx.x; i < ng * (kBN / 8); i += kConsumerThreads) {
        const int gr = i / (kBN / 8), c = i % (kBN / 8);
        zw[i] = (n0 + 8 * c < N) ? static_cast<uint32_t>(qz[size_t(g0 + gr) * (N / 8) + n0 / 8 + c]) : 0u;
      }
    }
    pdl_wait();
    // per-group sums of x over this CTA's k-range (deterministic warp reductions)
    for (int p = warp; p < MT * ng; p += kConsumerWarps) {
      const int m = p / ng, gi = p % ng, g = g0 + gi;
      const int kA = max(g * gsz, 32 * u0), kB = min((g + 1) * gsz, 32 * u1);
      float s = 0.f;
      if (m < M)
        for (int k = kA + lane; k < kB; k += 32) s += act_to_f32<ACT_BF16>(X[size_t(m) * K + k]);
      s = warp_sum(s);
      if (lane == 0) xg[m * a.ng_max + gi] = s;
    }
    consumer_sync(kConsumerThreads);

    float xnext[MT];
    auto load_x = [&](int u) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
        xnext[m] = (u < u1 && m < M) ? act_to_f32<ACT_BF16>(X[size_t(m) * K + 32 * u + lane]) * 256.f : 0.f;
    };
    load_x(u0 + warp);
    float2* myxs = xs + warp * MT * 32;
    const uint32_t magic = 0x3F000000u;

    for (int it = 0; it < n_loads; ++it) {
      const int s = it % kNS;
      const int u = u0 + it * kConsumerWarps + warp;
      const bool active = u < u1;
      __syncwarp();
#pragma unroll
      for (int m = 0; m < MT; ++m) myxs[m * 32 + lane] = make_float2(xnext[m], xnext[m]);
      __syncwarp();
      load_x(u + kConsumerWarps);
      if (!mbar_wait(&full[s], (it / kNS) & 1)) {
        *failed = 1;
        break;
      }
      if (active) {
        float2 accg[MT][2];
#pragma unroll
        for (int m = 0; m < MT; ++m) accg[m][0] = accg[m][1] = make_float2(0.f, 0.f);
        const uint8_t* rowp = stages + size_t(s) * kStageBytes + size_t(warp * kUnitRows) * (kBN * 4) + lane * 16;
#pragma unroll
        for (int i = 0; i < kUnitRows; ++i) {
          const uint4 wd = *reinterpret_cast<const uint4*>(rowp + i * (kBN * 4));
          const uint32_t w4[4] = {wd.x, wd.y, wd.z, wd.w};
          uint32_t lo[4], hi[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            lo[c] = w4[c] & 0x0F0F0F0Fu;
            hi[c] = (w4[c] >> 4) & 0x0F0F0F0Fu;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t sel = 0x7044u | (uint32_t(j >> 1) << 8);
            float mf[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) mf[c] = as_f32(prmt((j & 1) ? hi[c] : lo[c], magic, sel));
            const float2 m01 = make_float2(mf[0], mf[1]), m23 = make_float2(mf[2], mf[3]);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const float2 xp = myxs[m * 32 + 8 * i + j];
              accg[m][0] = ffma2(xp, m01, accg[m][0]);
              accg[m][1] = ffma2(xp, m23, accg[m][1]);
            }
          }
        }
        // fold the unit into the running sums with its group's scales
        const int gi = (32 * u) / gsz - g0;
        const uint2 sv = *reinterpret_cast<const uint2*>(scl + gi * kBN + lane * 4);
        const float s4[4] = {scale_bits_to_f32<ACT_BF16>(sv.x & 0xFFFFu), scale_bits_to_f32<ACT_BF16>(sv.x >> 16),
                             scale_bits_to_f32<ACT_BF16>(sv.y & 0xFFFFu), scale_bits_to_f32<ACT_BF16>(sv.y >> 16)};
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          acc[m][0] = fmaf(s4[0], accg[m][0].x, acc[m][0]);
          acc[m][1] = fmaf(s4[1], accg[m][0].y, acc[m][1]);
          acc[m][2] = fmaf(s4[2], accg[m][1].x, acc[m][2]);
          acc[m][3] = fmaf(s4[3], accg[m][1].y, acc[m][3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // cross-warp reduction (the stage ring is free: every issued load was consumed)
    consumer_sync(kConsumerThreads);
    float* red = reinterpret_cast<float*>(stages);
#pragma unroll
    for (int m = 0; m < MT; ++m)
      *reinterpret_cast<float4*>(red + (warp * MT + m) * kBN + lane * 4) =
          make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
    consumer_sync(kConsumerThreads);
    for (int e = threadIdx.x; e < MT * kBN; e += kConsumerThreads) {
      const int m = e / kBN, col = e % kBN;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) v += red[(w * MT + m) * kBN + col];
      // remove the 128 x offset of the codes and the zero points, per group
      float corr = 0.f;
      for (int gi = 0; gi < ng; ++gi) {
        const float sc = scale_bits_to_f32<ACT_BF16>(scl[gi * kBN + col]);
        const float z = HAS_Z ? float((zw[gi * (kBN / 8) + col / 8] >> (4 * (col % 8))) & 15u) : 8.f;
        corr = fmaf(sc * (128.f + z), xg[m * a.ng_max + gi], corr);
      }
      part[e] = v - corr;
    }
  }

  uint16_t* Y = static_cast<uint16_t*>(a.y);
  finish_tile<MT, kBN>(part, S, [&](int m, int col, float v) {
    const int n = n0 + col;
    if (m < M && n < N) Y[size_t(m) * N + n] = f32_to_act<ACT_BF16>(v);
  });
}

// ---------------------------------------------------------------------------
// Act-order: g(k) = g_idx[k], gathered per k from a {scale, offset} table.
// ---------------------------------------------------------------------------
template <int MT, int ACT_BF16, bool HAS_Z>
__global__ void __launch_bounds__(kGemvThreads, 1)
    k4g_gemv_kernel(const __grid_constant__ CUtensorMap wmap, const GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int G = a.K / a.group;
  const Smem4 L(MT, 0, true, G);
  uint8_t* stages = smem;
  float2* xs = reinterpret_cast<float2*>(smem + L.xs);
  uint32_t* goff = reinterpret_cast<uint32_t*>(smem + L.aux);                     // [8 warps][32]
  uint8_t* sd = smem + L.aux + size_t(kConsumerWarps) * 32 * 4;                    // [G][BN/2] x {s,s,d,d}
  float* part = reinterpret_cast<float*>(smem + L.part);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kNS;
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L.flag);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = gridDim.x, n0 = blockIdx.y * kBN;
  const int M = a.M, K = a.K, N = a.N;
  int u0, u1;
  split_range(K / 32, S, blockIdx.x, u0, u1);
  const int n_loads = (u1 - u0 + kConsumerWarps - 1) / kConsumerWarps;

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

  float2 acc[MT][2];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = make_float2(0.f, 0.f);

  if (warp == kConsumerWarps) {
    int issued = 0;
    if (lane == 0 && n_loads > 0)
      issued = produce_stages<kNS, kStageBytes>(&wmap, stages, full, empty, n0, 4 * u0, kStageRows, n_loads,
                                                failed);
    pdl_wait();
    if (lane == 0 && *failed) drain_stages<kNS>(full, issued);
  } else {
    const uint16_t* X = static_cast<const uint16_t*>(a.x);
    const uint16_t* SC = static_cast<const uint16_t*>(a.scales);
    const int32_t* QZ = static_cast<const int32_t*>(a.zeros);
    // {s0, s1, d0, d1} per column pair and group: d = -s (0.5 + z/256), exact in fp32
    for (int i = threadIdx.x; i < G * (kBN / 2); i += kConsumerThreads) {
      const int g = i / (kBN / 2), c = 2 * (i % (kBN / 2));
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (n0 + c < N) {
        const uint32_t sb = *reinterpret_cast<const uint32_t*>(SC + size_t(g) * N + n0 + c);
        const float s0 = scale_bits_to_f32<ACT_BF16>(sb & 0xFFFFu), s1 = scale_bits_to_f32<ACT_BF16>(sb >> 16);
        float z0 = 8.f, z1 = 8.f;
        if (HAS_Z) {
          const uint32_t zq = static_cast<uint32_t>(QZ[size_t(g) * (N / 8) + (n0 + c) / 8]);
          z0 = float((zq >> (4 * ((n0 + c) % 8))) & 15u);
          z1 = float((zq >> (4 * ((n0 + c + 1) % 8))) & 15u);
        }
        v = make_float4(s0, s1, -s0 * (0.5f + z0 * (1.f / 256.f)), -s1 * (0.5f + z1 * (1.f / 256.f)));
      }
      reinterpret_cast<float4*>(sd)[i] = v;
    }
    consumer_sync(kConsumerThreads);
    pdl_wait();

    float xnext[MT];
    uint32_t gnext = 0;
    auto load_x = [&](int u) {
      const bool ok = u < u1;
      if (ok) {
        int g = a.g_idx[32 * u + lane];
        g = min(max(g, 0), G - 1);  // out-of-range group indices are clamped, never read out of bounds
        gnext = uint32_t(g) * (kBN * 8);
      }
#pragma unroll
      for (int m = 0; m < MT; ++m)
        xnext[m] = (ok && m < M) ? act_to_f32<ACT_BF16>(X[size_t(m) * K + 32 * u + lane]) * 256.f : 0.f;
    };
    load_x(u0 + warp);
    float2* myxs = xs + warp * MT * 32;
    uint32_t* mygoff = goff + warp * 32;
    const uint32_t magic = 0x3F000000u;
    const uint32_t sd_lane = smem_u32(sd) + lane * 32;

    for (int it = 0; it < n_loads; ++it) {
      const int s = it % kNS;
      const int u = u0 + it * kConsumerWarps + warp;
      const bool active = u < u1;
      __syncwarp();
#pragma unroll
      for (int m = 0; m < MT; ++m) myxs[m * 32 + lane] = make_float2(xnext[m], xnext[m]);
      mygoff[lane] = gnext;
      __syncwarp();
      load_x(u + kConsumerWarps);
      if (!mbar_wait(&full[s], (it / kNS) & 1)) {
        *failed = 1;
        break;
      }
      if (active) {
        const uint8_t* rowp = stages + size_t(s) * kStageBytes + size_t(warp * kUnitRows) * (kBN * 4) + lane * 16;
#pragma unroll
        for (int i = 0; i < kUnitRows; ++i) {
          const uint4 wd = *reinterpret_cast<const uint4*>(rowp + i * (kBN * 4));
          const uint32_t w4[4] = {wd.x, wd.y, wd.z, wd.w};
          uint32_t lo[4], hi[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            lo[c] = w4[c] & 0x0F0F0F0Fu;
            hi[c] = (w4[c] >> 4) & 0x0F0F0F0Fu;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t sel = 0x7044u | (uint32_t(j >> 1) << 8);
            float mf[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) mf[c] = as_f32(prmt((j & 1) ? hi[c] : lo[c], magic, sel));
            const uint32_t row = sd_lane + mygoff[8 * i + j];
            const uint4 sd01 = lds128(row), sd23 = lds128(row + 16);
            const float2 w01 = ffma2(make_float2(as_f32(sd01.x), as_f32(sd01.y)), make_float2(mf[0], mf[1]),
                                     make_float2(as_f32(sd01.z), as_f32(sd01.w)));
            const float2 w23 = ffma2(make_float2(as_f32(sd23.x), as_f32(sd23.y)), make_float2(mf[2], mf[3]),
                                     make_float2(as_f32(sd23.z), as_f32(sd23.w)));
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const float2 xp = myxs[m * 32 + 8 * i + j];
              acc[m][0] = ffma2(xp, w01, acc[m][0]);
              acc[m][1] = ffma2(xp, w23, acc[m][1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    consumer_sync(kConsumerThreads);
    float* red = reinterpret_cast<float*>(stages);
#pragma unroll
    for (int m = 0; m < MT; ++m)
      *reinterpret_cast<float4*>(red + (warp * MT + m) * kBN + lane * 4) =
          make_float4(acc[m][0].x, acc[m][0].y, acc[m][1].x, acc[m][1].y);
    consumer_sync(kConsumerThreads);
    for (int e = threadIdx.x; e < MT * kBN; e += kConsumerThreads) {
      const int m = e / kBN, col = e % kBN;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) v += red[(w * MT + m) * kBN + col];
      part[e] = v;
    }
  }

  uint16_t* Y = static_cast<uint16_t*>(a.y);
  finish_tile<MT, kBN>(part, S, [&](int m, int col, float v) {
    const int n = n0 + col;
    if (m < M && n < N) Y[size_t(m) * N + n] = f32_to_act<ACT_BF16>(v);
  });
}

template <int MT, int ACT, bool HZ, bool AO>
void launch_one(const LaunchPlan& p, const CUtensorMap& map, const GemvArgs& a, cudaError_t& err) {
  auto kern = AO ? k4g_gemv_kernel<MT, ACT, HZ> : k4_gemv_kernel<MT, ACT, HZ>;
  const Smem4 L(MT, a.ng_max, AO, a.K / a.group);
  err = launch_gemv_kernel(reinterpret_cast<const void*>(kern), p, L.total, map, a);
}

template <int MT>
void dispatch_act(const LaunchPlan& p, const CUtensorMap& map, const GemvArgs& a, int act_bf16, bool has_z,
                  bool act_order, cudaError_t& err) {
  if (act_bf16) {
    if (has_z) { if (act_order) launch_one<MT, 1, true, true>(p, map, a, err); else launch_one<MT, 1, true, false>(p, map, a, err); }
    else       { if (act_order) launch_one<MT, 1, false, true>(p, map, a, err); else launch_one<MT, 1, false, false>(p, map, a, err); }
  } else {
    if (has_z) { if (act_order) launch_one<MT, 0, true, true>(p, map, a, err); else launch_one<MT, 0, true, false>(p, map, a, err); }
    else       { if (act_order) launch_one<MT, 0, false, true>(p, map, a, err); else launch_one<MT, 0, false, false>(p, map, a, err); }
  }
}

}  // namespace

size_t wq4_gemv_smem_bytes(int MT, int ng_max, bool act_order, int G) {
  return Smem4(MT, ng_max, act_order, G).total;
}

cudaError_t launch_wq4_gemv(const LaunchPlan& p, const CUtensorMap& map, const GemvArgs& a, int act_bf16,
                            bool has_z, bool act_order) {
  cudaError_t err = cudaErrorInvalidValue;
  switch (p.MT) {
    case 1: dispatch_act<1>(p, map, a, act_bf16, has_z, act_order, err); break;
    case 2: dispatch_act<2>(p, map, a, act_bf16, has_z, act_order, err); break;
    case 4: dispatch_act<4>(p, map, a, act_bf16, has_z, act_order, err); break;
    case 8: dispatch_act<8>(p, map, a, act_bf16, has_z, act_order, err); break;
    default: break;
  }
  return err;
}

}  // namespace wq
