// wq_gemv4.cu -- 4-bit group-wise weight-only GEMV / skinny GEMM on CUDA cores
// (M <= 8), with contiguous groups or act-order (g_idx).
//
// Definition ("Quantization CUDA", Weight Only Quantization / 量化粒度 and
// Marlin 格式):  y[m,n] = sum_k x[m,k] * s[g(k),n] * (q(k,n) - z[g(k),n]).
// Storage: qweight int32 [K/8, N], nibble j of word [r, n] = code of row 8r+j
// ("Int4 Weight Only Quantization / Weight Store": codes consecutive along K).
//
// Exact code conversion.  PRMT places a nibble q (0..15, high nibble already
// cleared) in byte 2 of the word 0x3F000000, which is the fp32 value
// m = 0.5 + q/256 exactly.  With x' = 256 x (exact), x' m = 128 x + x q is an
// exact product (at most 19 significant bits), so the only rounding is the
// fp32 accumulation.  The 128 x term is removed where the scale is applied:
//   contiguous groups, per 32-value unit u of group g:
//       y += s_g * (sum_{k in u} x'_k m_k - (128 + z_g) X_u),  X_u = sum_{k in u} x_k
//   act-order: w = fma(s, m, d) with d = -s (0.5 + z/256) is exactly
//       s (q - z) / 256, and y += x' w for every code.
#include "wq_gemv_common.cuh"
#include "wq_launch.h"

namespace wq {
namespace {

constexpr int kBN = 128;          // columns per tile (one 512-byte row per warp)
constexpr int kUnitRows = 4;      // packed rows per consumer unit (32 values of k)
constexpr int kStageRows = kConsumerWarps * kUnitRows;
constexpr int kStageK = kStageRows * 8;            // 256 values of k per stage
constexpr int kStageBytes = kStageRows * kBN * 4;  // 16 KB
constexpr int kNS = 3;  // two CTAs (bound by registers) leave room on the SM for the next kernel's first CTA

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

// Shared-memory carve-up (same arithmetic on host and device).
struct Smem4 {
  size_t xst, xc, aux, zw, xfull, recv, bars, flag, total;
  // xfull_bytes: the whole x (MT rows of K values) for the permuted variant, else 0
  __host__ __device__ Smem4(int MT, int ng_max, bool act_order, int G, int S, size_t xfull_bytes = 0) {
    size_t o = size_t(kNS) * kStageBytes;
    // raw x (or the perm slice of the sorted variant) per stage, then g_idx per stage for act-order
    xst = o;  o = align16(o + size_t(kNS) * (MT * kStageK * 2 > kStageK * 4 ? MT * kStageK * 2 : kStageK * 4));
    if (act_order) o = align16(o + size_t(kNS) * kStageK * 4);
    xc = o;   o = align16(o + size_t(MT) * kStageK * 8);                  // converted x pairs
    aux = o;  // contiguous: raw 16-bit scales [ng_max][BN]; act-order: goff [256] + sd [G][2][32][4] floats
    if (act_order) o = align16(o + size_t(kStageK) * 4 + size_t(G) * kBN * 8);
    else           o = align16(o + size_t(ng_max) * kBN * 2);
    zw = o;   o = align16(o + (act_order ? 0 : size_t(ng_max) * (kBN / 8) * 4));
    xfull = o; o = align16(o + xfull_bytes);
    recv = o; o = align16(o + TileReduce(S, kBN).recv_floats(MT) * 4);
    bars = o; o = align16(o + size_t(2 * kNS + 1) * 8);
    flag = o; o = align16(o + 16);
    total = o;
  }
};

template <int ACT_BF16>
__device__ __forceinline__ float scale_bits_to_f32(uint32_t bits16) {
  return ACT_BF16 ? bf16_bits_to_f32(bits16) : f16_bits_to_f32(bits16);
}

// Unpack one 512-byte row slice (4 columns x 8 codes) and accumulate
// x' * m into acc[m][0] (columns 0,1) and acc[m][1] (columns 2,3).
template <int MT>
__device__ __forceinline__ void unit_row_accumulate(uint4 wd, const float4* xrow /* [MT] stride kStageK/2 */,
                                                    float2 (*acc)[2]) {
  const uint32_t w4[4] = {wd.x, wd.y, wd.z, wd.w};
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    lo[c] = w4[c] & 0x0F0F0F0Fu;
    hi[c] = (w4[c] >> 4) & 0x0F0F0F0Fu;
  }
  float4 xq[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int p = 0; p < 4; ++p) xq[m][p] = xrow[m * (kStageK / 2) + p];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t sel = 0x7044u | (uint32_t(j >> 1) << 8);
    const uint32_t* src = (j & 1) ? hi : lo;
    const float2 m01 = make_float2(as_f32(prmt(src[0], 0x3F000000u, sel)), as_f32(prmt(src[1], 0x3F000000u, sel)));
    const float2 m23 = make_float2(as_f32(prmt(src[2], 0x3F000000u, sel)), as_f32(prmt(src[3], 0x3F000000u, sel)));
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float4 q = xq[m][j >> 1];
      const float2 xp = (j & 1) ? make_float2(q.z, q.w) : make_float2(q.x, q.y);
      acc[m][0] = ffma2(xp, m01, acc[m][0]);
      acc[m][1] = ffma2(xp, m23, acc[m][1]);
    }
  }
}

// ---------------------------------------------------------------------------
// Contiguous groups (g(k) = k / group).  PERM: the weight rows were sorted by
// act-order group once ahead of time (wq4_actorder_prepare); row i of the
// sorted weights multiplies x[perm[i]].  The whole x then sits in shared
// memory and each stage brings the slice of perm (TMA box of the "x" map).
// ---------------------------------------------------------------------------
template <int MT, int ACT_BF16, bool HAS_Z, bool PERM>
__global__ void __launch_bounds__(kGemvThreads, 1)
    k4_gemv_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                   const GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Smem4 L(MT, a.ng_max, false, 0, gridDim.x, PERM ? size_t(MT) * a.K * 2 : 0);
  const TileReduce R(gridDim.x, kBN);
  const uint16_t* xfull = reinterpret_cast<const uint16_t*>(smem + L.xfull);
  uint8_t* wst = smem;
  uint8_t* xst = smem + L.xst;
  float2* xc = reinterpret_cast<float2*>(smem + L.xc);
  uint16_t* scl = reinterpret_cast<uint16_t*>(smem + L.aux);
  uint32_t* zw = reinterpret_cast<uint32_t*>(smem + L.zw);
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kNS;
  uint64_t* recv_bar = empty + kNS;
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L.flag);       // producer's
  volatile int* cfailed = failed + 1;                                            // consumers'

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = gridDim.x, n0 = blockIdx.y * kBN;
  const int M = a.M, K = a.K, N = a.N, gsz = a.group;
  int u0, u1;
  split_range(K / 32, S, blockIdx.x, u0, u1);
  const int n_loads = (u1 - u0 + kConsumerWarps - 1) / kConsumerWarps;
  const UnitGroups ug(gsz, 32);
  const int g0 = ug.of(u0);
  const int ng = (u1 > u0) ? (32 * u1 - 1) / gsz - g0 + 1 : 0;

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
      issued = produce_stages<kNS>(&wmap, &xmap, wst, kStageBytes, xst, PERM ? kStageK * 4 : MT * kStageK * 2, full,
                                   empty, n0, 4 * u0, kStageRows, 32 * u0, kStageK, n_loads, failed);
    pdl_wait();
    if (lane == 0 && *failed) drain_stages<kNS>(full, issued);
    __syncwarp();
    if (S > 1) cluster_wait();
  } else {
    const int tid = threadIdx.x;
    // scale (and zero) slice of this CTA: weight-side data, read before the dependency wait
    for (int i = tid; i < ng * (kBN / 2); i += kConsumerThreads) {
      const int gr = i / (kBN / 2), c = 2 * (i % (kBN / 2));
      uint32_t v = 0;
      if (n0 + c < N)
        v = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(a.scales) + size_t(g0 + gr) * N + n0 + c);
      reinterpret_cast<uint32_t*>(scl)[i] = v;
    }
    if (HAS_Z) {
      const int32_t* qz = static_cast<const int32_t*>(a.zeros);
      for (int i = tid; i < ng * (kBN / 8); i += kConsumerThreads) {
        const int gr = i / (kBN / 8), c = i % (kBN / 8);
        zw[i] = (n0 + 8 * c < N) ? static_cast<uint32_t>(qz[size_t(g0 + gr) * (N / 8) + n0 / 8 + c]) : 0u;
      }
    }
    pdl_wait();
    consumer_sync(kConsumerThreads);  // the scale and zero tables are complete before any warp folds
    if (PERM) {  // the whole x in shared memory (rows >= M read as zero)
      uint4* xf = reinterpret_cast<uint4*>(smem + L.xfull);
      const int chunks_per_row = K / 8;
      for (int i = tid; i < MT * chunks_per_row; i += kConsumerThreads) {
        const int m = i / chunks_per_row, c = i % chunks_per_row;
        xf[i] = (m < M) ? reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + size_t(m) * K)[c]
                        : make_uint4(0u, 0u, 0u, 0u);
      }
      consumer_sync(kConsumerThreads);
    }

    float2 acc[MT][2];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = make_float2(0.f, 0.f);

    float2* xcw = xc + warp * 32;  // this warp's x pairs: [MT][stride kStageK]
    for (int it = 0; it < n_loads; ++it) {
      const int s = it % kNS;
      const int u = u0 + it * kConsumerWarps + warp;
      if (!mbar_wait(&full[s], (it / kNS) & 1)) *cfailed = 1;
      if (*cfailed) break;
      // convert this warp's 32 values of x (one per lane, every row)
      float xu[MT];
      {
        const uint16_t* xr = reinterpret_cast<const uint16_t*>(xst + size_t(s) * MT * kStageK * 2) + warp * 32 + lane;
        int kp = 0;
        if (PERM) {
          kp = reinterpret_cast<const int32_t*>(xst + size_t(s) * kStageK * 4)[warp * 32 + lane];
          kp = min(max(kp, 0), K - 1);  // out-of-range entries are clamped, never read out of bounds
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const float v = act_to_f32<ACT_BF16>(PERM ? xfull[size_t(m) * K + kp] : xr[m * kStageK]);
          xcw[m * kStageK + lane] = make_float2(v * 256.f, v * 256.f);
          xu[m] = warp_sum(v);  // X_u of this warp's unit
        }
      }
      __syncwarp();
      if (u < u1) {
        float2 accg[MT][2];
#pragma unroll
        for (int m = 0; m < MT; ++m) accg[m][0] = accg[m][1] = make_float2(0.f, 0.f);
        const uint8_t* rowp = wst + size_t(s) * kStageBytes + size_t(warp * kUnitRows) * (kBN * 4) + lane * 16;
        const float4* xw = reinterpret_cast<const float4*>(xcw);
#pragma unroll
        for (int i = 0; i < kUnitRows; ++i)
          unit_row_accumulate<MT>(*reinterpret_cast<const uint4*>(rowp + i * (kBN * 4)), xw + 4 * i, accg);
        // apply the unit's group scale, removing the 128 x offset and the zero point
        const int gi = ug.of(u) - g0;
        const uint2 sv = *reinterpret_cast<const uint2*>(scl + gi * kBN + lane * 4);
        const float2 s01 = make_float2(scale_bits_to_f32<ACT_BF16>(sv.x & 0xFFFFu), scale_bits_to_f32<ACT_BF16>(sv.x >> 16));
        const float2 s23 = make_float2(scale_bits_to_f32<ACT_BF16>(sv.y & 0xFFFFu), scale_bits_to_f32<ACT_BF16>(sv.y >> 16));
        float2 c01 = make_float2(-136.f, -136.f), c23 = c01;
        if (HAS_Z) {
          const uint32_t zq = zw[gi * (kBN / 8) + lane / 2] >> (16 * (lane & 1));
          c01 = make_float2(-128.f - float(zq & 15u), -128.f - float((zq >> 4) & 15u));
          c23 = make_float2(-128.f - float((zq >> 8) & 15u), -128.f - float((zq >> 12) & 15u));
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const float2 xx = make_float2(xu[m], xu[m]);
          acc[m][0] = ffma2(s01, ffma2(c01, xx, accg[m][0]), acc[m][0]);
          acc[m][1] = ffma2(s23, ffma2(c23, xx, accg[m][1]), acc[m][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    push_partials<MT, kBN>(R, acc, recv, recv_bar, warp, lane);
  }

  uint16_t* Y = static_cast<uint16_t*>(a.y);
  owner_reduce_store<MT, kBN>(R, recv, recv_bar, [&](int m, int col, float v) {
    const int n = n0 + col;
    if (m < M && n < N) Y[size_t(m) * N + n] = f32_to_act<ACT_BF16>(v);
  });
}

// ---------------------------------------------------------------------------
// Act-order: g(k) = g_idx[k], gathered per k from a {scale, offset} table laid
// out so that a warp reads one contiguous 512-byte half-row per load.
// ---------------------------------------------------------------------------
template <int MT, int ACT_BF16, bool HAS_Z>
__global__ void __launch_bounds__(kGemvThreads, 1)
    k4g_gemv_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                    const __grid_constant__ CUtensorMap gmap, const GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int G = a.K / a.group;
  const Smem4 L(MT, 0, true, G, gridDim.x);
  const TileReduce R(gridDim.x, kBN);
  uint8_t* wst = smem;
  uint8_t* xst = smem + L.xst;
  uint8_t* gst = smem + L.xst + size_t(kNS) * (MT * kStageK * 2 > kStageK * 4 ? MT * kStageK * 2 : kStageK * 4);
  float2* xc = reinterpret_cast<float2*>(smem + L.xc);
  uint32_t* goff = reinterpret_cast<uint32_t*>(smem + L.aux);        // [256] byte offsets of sd rows
  uint8_t* sd = smem + L.aux + size_t(kStageK) * 4;                  // [G][2 halves][32 lanes] x float4
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kNS;
  uint64_t* recv_bar = empty + kNS;
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L.flag);       // producer's
  volatile int* cfailed = failed + 1;                                            // consumers'

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = gridDim.x, n0 = blockIdx.y * kBN;
  const int M = a.M, K = a.K, N = a.N;
  int u0, u1;
  split_range(K / 32, S, blockIdx.x, u0, u1);
  const int n_loads = (u1 - u0 + kConsumerWarps - 1) / kConsumerWarps;
  constexpr uint32_t kXBytes = MT * kStageK * 2, kGBytes = kStageK * 4;

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
    if (lane == 0 && n_loads > 0) {
      prefetch_tensormap(&wmap);
      prefetch_tensormap(&xmap);
      prefetch_tensormap(&gmap);
      const uint64_t pol = l2_evict_first_policy();
      const int pre = n_loads < kNS ? n_loads : kNS;
      for (int it = 0; it < pre; ++it) {
        mbar_expect_tx(&full[it], kStageBytes + kXBytes + kGBytes);
        tma_load_2d(wst + size_t(it) * kStageBytes, &wmap, &full[it], n0, 4 * u0 + it * kStageRows, pol);
        tma_load_2d(gst + size_t(it) * kGBytes, &gmap, &full[it], 32 * u0 + it * kStageK, 0, 0ull);
      }
      pdl_wait();
      for (int it = 0; it < pre; ++it)
        tma_load_2d(xst + size_t(it) * kXBytes, &xmap, &full[it], 32 * u0 + it * kStageK, 0, 0ull);
      issued = pre;
      for (int it = kNS; it < n_loads; ++it) {
        const int s = it % kNS;
        if (*failed || !mbar_wait(&empty[s], ((it / kNS) - 1) & 1)) {
          *failed = 1;
          break;
        }
        mbar_expect_tx(&full[s], kStageBytes + kXBytes + kGBytes);
        tma_load_2d(wst + size_t(s) * kStageBytes, &wmap, &full[s], n0, 4 * u0 + it * kStageRows, pol);
        tma_load_2d(gst + size_t(s) * kGBytes, &gmap, &full[s], 32 * u0 + it * kStageK, 0, 0ull);
        tma_load_2d(xst + size_t(s) * kXBytes, &xmap, &full[s], 32 * u0 + it * kStageK, 0, 0ull);
        ++issued;
      }
    }
    pdl_wait();
    if (lane == 0 && *failed) drain_stages<kNS>(full, issued);
    __syncwarp();
    if (S > 1) cluster_wait();
  } else {
    const int tid = threadIdx.x;
    const uint16_t* SC = static_cast<const uint16_t*>(a.scales);
    const int32_t* QZ = static_cast<const int32_t*>(a.zeros);
    // table row g: half h, lane l -> {s(c0), s(c0+1), d(c0), d(c0+1)}, c0 = 4l + 2h,
    // d = -s (0.5 + z/256) (exact in fp32)
    for (int i = tid; i < G * (kBN / 2); i += kConsumerThreads) {
      const int g = i / (kBN / 2), r = i % (kBN / 2), h = r / 32, l = r % 32;
      const int c = 4 * l + 2 * h;
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
    pdl_wait();
    consumer_sync(kConsumerThreads);  // the table is complete before any warp gathers from it

    float2 acc[MT][2];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = make_float2(0.f, 0.f);
    const uint32_t sd_lane = smem_u32(sd) + lane * 16;

    float2* xcw = xc + warp * 32;
    uint32_t* gw_own = goff + warp * 32;
    for (int it = 0; it < n_loads; ++it) {
      const int s = it % kNS;
      const int u = u0 + it * kConsumerWarps + warp;
      if (!mbar_wait(&full[s], (it / kNS) & 1)) *cfailed = 1;
      if (*cfailed) break;
      {
        const uint16_t* xr = reinterpret_cast<const uint16_t*>(xst + size_t(s) * kXBytes) + warp * 32 + lane;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const float v = act_to_f32<ACT_BF16>(xr[m * kStageK]) * 256.f;
          xcw[m * kStageK + lane] = make_float2(v, v);
        }
        int g = reinterpret_cast<const int32_t*>(gst + size_t(s) * kGBytes)[warp * 32 + lane];
        g = min(max(g, 0), G - 1);  // out-of-range group indices are clamped, never read out of bounds
        gw_own[lane] = uint32_t(g) * (kBN * 8);
      }
      __syncwarp();
      if (u < u1) {
        const uint8_t* rowp = wst + size_t(s) * kStageBytes + size_t(warp * kUnitRows) * (kBN * 4) + lane * 16;
        const float4* xw = reinterpret_cast<const float4*>(xcw);
        const uint4* gw = reinterpret_cast<const uint4*>(gw_own);
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
          const uint4 go0 = gw[2 * i], go1 = gw[2 * i + 1];
          const uint32_t gofs[8] = {go0.x, go0.y, go0.z, go0.w, go1.x, go1.y, go1.z, go1.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t sel = 0x7044u | (uint32_t(j >> 1) << 8);
            const uint32_t* src = (j & 1) ? hi : lo;
            const float2 m01 = make_float2(as_f32(prmt(src[0], 0x3F000000u, sel)), as_f32(prmt(src[1], 0x3F000000u, sel)));
            const float2 m23 = make_float2(as_f32(prmt(src[2], 0x3F000000u, sel)), as_f32(prmt(src[3], 0x3F000000u, sel)));
            const uint32_t row = sd_lane + gofs[j];
            const uint4 t01 = lds128(row), t23 = lds128(row + 512);
            const float2 w01 = ffma2(make_float2(as_f32(t01.x), as_f32(t01.y)), m01, make_float2(as_f32(t01.z), as_f32(t01.w)));
            const float2 w23 = ffma2(make_float2(as_f32(t23.x), as_f32(t23.y)), m23, make_float2(as_f32(t23.z), as_f32(t23.w)));
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const float4 q = xw[m * (kStageK / 2) + 4 * i + (j >> 1)];
              const float2 xp = (j & 1) ? make_float2(q.z, q.w) : make_float2(q.x, q.y);
              acc[m][0] = ffma2(xp, w01, acc[m][0]);
              acc[m][1] = ffma2(xp, w23, acc[m][1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    push_partials<MT, kBN>(R, acc, recv, recv_bar, warp, lane);
  }

  uint16_t* Y = static_cast<uint16_t*>(a.y);
  owner_reduce_store<MT, kBN>(R, recv, recv_bar, [&](int m, int col, float v) {
    const int n = n0 + col;
    if (m < M && n < N) Y[size_t(m) * N + n] = f32_to_act<ACT_BF16>(v);
  });
}

cudaError_t launch3(const void* kern, const LaunchPlan& p, size_t smem, const CUtensorMap& w, const CUtensorMap& x,
                    const CUtensorMap* g, const GemvArgs& a) {
  const CUtensorMap* maps[3] = {&w, &x, g};
  return launch_gemv_kernel(kern, p, smem, maps, g ? 3 : 2, a);
}

// mode 0: contiguous groups, 1: act-order gather (g = g_idx map), 2: sorted rows (x = perm map)
template <int MT, int ACT, bool HZ>
cudaError_t launch_one(const LaunchPlan& p, const CUtensorMap& w, const CUtensorMap& x, const CUtensorMap* g,
                       const GemvArgs& a, int mode) {
  if (mode == 1)
    return launch3(reinterpret_cast<const void*>(k4g_gemv_kernel<MT, ACT, HZ>), p,
                   Smem4(MT, a.ng_max, true, a.K / a.group, p.S).total, w, x, g, a);
  if (mode == 2)
    return launch3(reinterpret_cast<const void*>(k4_gemv_kernel<MT, ACT, HZ, true>), p,
                   Smem4(MT, a.ng_max, false, 0, p.S, size_t(MT) * a.K * 2).total, w, x, nullptr, a);
  return launch3(reinterpret_cast<const void*>(k4_gemv_kernel<MT, ACT, HZ, false>), p,
                 Smem4(MT, a.ng_max, false, 0, p.S).total, w, x, nullptr, a);
}

template <int MT>
cudaError_t dispatch_act(const LaunchPlan& p, const CUtensorMap& w, const CUtensorMap& x, const CUtensorMap* g,
                         const GemvArgs& a, int act_bf16, bool has_z, int mode) {
  if (act_bf16) return has_z ? launch_one<MT, 1, true>(p, w, x, g, a, mode) : launch_one<MT, 1, false>(p, w, x, g, a, mode);
  return has_z ? launch_one<MT, 0, true>(p, w, x, g, a, mode) : launch_one<MT, 0, false>(p, w, x, g, a, mode);
}

}  // namespace

size_t wq4_gemv_smem_bytes(int MT, int ng_max, bool act_order, int G, int S, size_t xfull_bytes) {
  return Smem4(MT, ng_max, act_order, G, S, xfull_bytes).total;
}

int wq4_stage_k() { return kStageK; }

cudaError_t launch_wq4_gemv(const LaunchPlan& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                            const CUtensorMap* gmap, const GemvArgs& a, int act_bf16, bool has_z, bool sorted) {
  const int mode = gmap ? 1 : (sorted ? 2 : 0);
  switch (p.MT) {
    case 1: return dispatch_act<1>(p, wmap, xmap, gmap, a, act_bf16, has_z, mode);
    case 2: return dispatch_act<2>(p, wmap, xmap, gmap, a, act_bf16, has_z, mode);
    case 4: return dispatch_act<4>(p, wmap, xmap, gmap, a, act_bf16, has_z, mode);
    case 8: return dispatch_act<8>(p, wmap, xmap, gmap, a, act_bf16, has_z, mode);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace wq
