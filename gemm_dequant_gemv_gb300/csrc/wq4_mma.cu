// wq4_mma.cu -- 4-bit group-wise weight-only GEMM for M > 8 on the tcgen05
// tensor cores (M up to 64 per launch; larger M runs in 64-row chunks).
//
// Definition ("Quantization CUDA", 量化粒度 and Marlin 格式):
//   y[m,n] = sum_g s[g,n] * sum_{k in g} x[m,k] * (q(k,n) - z[g,n]).
// The weight side is the MMA's M dimension (swap-AB): one CTA owns 128 output
// columns, D[n, m] lives in tensor memory (128 lanes x Mp fp32 columns).
//
// Per k-stage of KS = 128 values (64 when the group size is not a multiple of
// 128):
//   * warp 8 (TMA) loads the packed int32 words [KS/8 rows x 128 columns] and
//     the x tile [Mp rows x KS] (128-byte-swizzled boxes of 64 values) into a
//     ring of stages;
//   * warps 0-3 (converters, one output column per thread = one tensor-memory
//     lane) unpack the nibbles to the exact 16-bit integers q - z (PRMT into
//     128 + q / 1024 + q, then one packed subtraction) and store them with
//     tcgen05.st as the A operand in tensor memory (fp16 pairs of consecutive k
//     per 32-bit column), so the dequantized weights never touch shared memory;
//   * warp 9 issues KS/16 kind::f16 MMAs (K = 16 each, A from tensor memory,
//     B = x from shared memory) per stage into one of two tensor-memory
//     accumulators, one accumulator per scale group;
//   * warps 4-7 (epilogue) drain each finished group accumulator and apply the
//     group's scale in fp32: y += s[g,n] * D_g[n,:].
// Products (q - z) * x are exact; the only roundings are the fp32 sums.  The K
// slices of a column tile form a thread-block cluster that reduces through
// distributed shared memory, as in the CUDA-core kernels.
#include <algorithm>

#include "../../include/wq.h"
#include "wq_gemv_common.cuh"
#include "wq_mma.h"
#include "wq_tcgen05.cuh"

namespace wq {

bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swizzle);
int device_sm_count();
int device_max_smem();

namespace {

constexpr int kBN = 128;            // output columns per tile (MMA M)
constexpr int kBoxK = 64;           // values of k per 128-byte-swizzled x box
constexpr int kNA = 2;              // dequantized A stages in tensor memory
constexpr int kWarpTMA = 8, kWarpMMA = 9;
constexpr int kThreads = 10 * 32;
constexpr int kPf = 8;              // scale groups whose scales / zeros are fetched ahead

// Per-KS constants: stages in the TMA ring, bytes of packed weights per stage,
// and the tensor-memory columns (two group accumulators, then the A stages).
template <int KS> struct Stage {
  static constexpr int NS = KS == 64 ? 6 : 4;
  static constexpr int kPacked = (KS / 8) * kBN * 4;  // 4 or 8 KB
  static constexpr uint32_t kACols = KS / 2;           // fp16 pairs per A stage
};
template <int MP, int KS> struct Tmem {
  static constexpr uint32_t kA = 2 * MP;               // first A column
  static constexpr uint32_t kUsed = 2 * MP + kNA * Stage<KS>::kACols;
  static constexpr uint32_t kCols = kUsed <= 32 ? 32 : kUsed <= 64 ? 64 : kUsed <= 128 ? 128 : kUsed <= 256 ? 256 : 512;
  static_assert(kUsed <= 256, "two CTAs per SM share the 512 tensor-memory columns");
};

struct MmaArgs {
  void* y;
  const void* scales;
  const int32_t* qzeros;
  int M, K, N, group;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) & ~(a - 1); }

struct SmemMma {
  size_t xs, pw, part, bars, misc, total;
  __host__ __device__ SmemMma(int MP, int KS) {
    const int NS = KS == 64 ? Stage<64>::NS : Stage<128>::NS;
    size_t o = 0;
    xs = o;   o += size_t(NS) * MP * KS * 2;            // x stages (boxes of Mp x 64, 1024-byte multiples)
    pw = o;   o += size_t(NS) * (KS / 8) * kBN * 4;
    part = o; o = align_up(o + size_t(MP) * kBN * 4, 16);
    bars = o; o = align_up(o + size_t(2 * NS + 2 * kNA + 4) * 8, 16);
    misc = o; o = align_up(o + 32, 16);
    total = o + 1024;  // slack to align the base to 1024 bytes
  }
};

template <int ACT_BF16>
__device__ __forceinline__ uint32_t sub2(uint32_t a, uint32_t b) {
  uint32_t d;
  if (ACT_BF16)
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <int MP, int ACT_BF16, bool HAS_Z, int KS>
__global__ void __launch_bounds__(kThreads, MP <= 32 ? 2 : 1)  // two CTAs per SM up to Mp = 32
    wq4_mma_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                   const MmaArgs a) {
  constexpr int kNS = Stage<KS>::NS;
  constexpr int kPackedStageBytes = Stage<KS>::kPacked;
  constexpr uint32_t kACols = Stage<KS>::kACols;
  constexpr int kXStageBytes = MP * KS * 2;
  constexpr int kXBoxBytes = MP * kBoxK * 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemMma L(MP, KS);
  uint8_t* sX = smem + L.xs;
  uint8_t* sW = smem + L.pw;
  float* part = reinterpret_cast<float*>(smem + L.part);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kNS;
  uint64_t* a_full = empty + kNS;
  uint64_t* a_empty = a_full + kNA;
  uint64_t* t_full = a_empty + kNA;
  uint64_t* t_empty = t_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L.misc + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = gridDim.x, n0 = blockIdx.y * kBN;
  const int M = a.M, K = a.K, N = a.N, gsz = a.group;
  const int spg = gsz / KS;  // stages per group
  int g0, g1;
  split_range(K / gsz, S, blockIdx.x, g0, g1);
  const int ng = g1 - g0, nst = ng * spg, ks0 = g0 * spg;
  constexpr uint32_t kTmemCols = Tmem<MP, KS>::kCols;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kNA; ++s) {
      mbar_init(&a_full[s], 4);  // one arrival per converter warp
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&t_full[s], 1);
      mbar_init(&t_empty[s], 4);  // one arrival per epilogue warp
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

  float acc[MP];
#pragma unroll
  for (int m = 0; m < MP; ++m) acc[m] = 0.f;

  if (warp == kWarpTMA) {
    // ------------------------------------------------------------ producer --
    // The boxes of a stage are issued by different lanes (lane 0: the packed
    // weights, lanes 1 ..: the x boxes): on GB300 each issuing thread moves at
    // most about three million TMA boxes per second (measured), so a single
    // thread issuing all of them bounded the whole kernel.
    if (nst > 0) {
      if (lane == 0) {
        prefetch_tensormap(&wmap);
        prefetch_tensormap(&xmap);
      }
      const uint64_t pol = l2_evict_first_policy();
      const uint32_t stage_bytes = kPackedStageBytes + kXStageBytes;
      const int pre = nst < kNS ? nst : kNS;
      // weights of the first stages before the dependency wait, x after it
      for (int i = 0; i < pre; ++i) {
        if (lane == 0) mbar_expect_tx(&full[i], stage_bytes);
        __syncwarp();
        if (lane == 0) tma_load_2d(sW + size_t(i) * kPackedStageBytes, &wmap, &full[i], n0, (ks0 + i) * (KS / 8), pol);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i)
        if (lane >= 1 && lane <= KS / kBoxK) {
          const int h = lane - 1;
          tma_load_2d(sX + size_t(i) * kXStageBytes + h * kXBoxBytes, &xmap, &full[i], (ks0 + i) * KS + h * kBoxK, 0, 0ull);
        }
      for (int i = kNS; i < nst; ++i) {
        const int s = i % kNS;
        if (lane == 0) {
          if (*failed || !mbar_wait_sleep(&empty[s], ((i / kNS) - 1) & 1)) *failed = 1;
          else mbar_expect_tx(&full[s], stage_bytes);
        }
        __syncwarp();
        if (*failed) break;
        if (lane == 0) {
          tma_load_2d(sW + size_t(s) * kPackedStageBytes, &wmap, &full[s], n0, (ks0 + i) * (KS / 8), pol);
        } else if (lane <= KS / kBoxK) {
          const int h = lane - 1;
          tma_load_2d(sX + size_t(s) * kXStageBytes + h * kXBoxBytes, &xmap, &full[s], (ks0 + i) * KS + h * kBoxK, 0, 0ull);
        }
      }
    } else {
      pdl_wait();
    }
  } else if (warp == kWarpMMA) {
    // ----------------------------------------------------------------- MMA --
    pdl_wait();
    if (lane == 0) {
      const uint32_t idesc = f16_idesc(kBN, MP, ACT_BF16);
      int last = -1;
      for (int i = 0; i < nst; ++i) {
        const int s = i % kNS, ab = i % kNA, gi = i / spg, tb = gi & 1;
        if (i % spg == 0 && gi >= 2) {
          if (!mbar_wait_sleep(&t_empty[tb], ((gi / 2) - 1) & 1)) { *failed = 1; break; }
        }
        if (!mbar_wait_sleep(&a_full[ab], (i / kNA) & 1) || !mbar_wait_sleep(&full[s], (i / kNS) & 1)) {
          *failed = 1;
          break;
        }
        tc_fence_after();
        const uint32_t acol = tmem + Tmem<MP, KS>::kA + ab * kACols;
        const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sX + size_t(s) * kXStageBytes));
#pragma unroll
        for (int k = 0; k < KS / 16; ++k)
          mma_f16_ts(tmem + tb * MP, acol + 8 * k,
                     bdesc + uint64_t(((k / (kBoxK / 16)) * kXBoxBytes + 32 * (k % (kBoxK / 16))) >> 4), idesc,
                     (i % spg != 0 || k > 0) ? 1u : 0u);
        mma_commit(&empty[s]);
        mma_commit(&a_empty[ab]);
        if (i % spg == spg - 1) mma_commit(&t_full[tb]);
        last = i;
      }
      // the tensor memory is released only after the last MMA has completed
      if (last >= 0) mbar_wait_sleep(&empty[last % kNS], (last / kNS) & 1);
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------- converters --
    const int col = threadIdx.x;  // 0..127
    const int n = n0 + col;
    const uint32_t magic = ACT_BF16 ? 0x43434343u : 0x64646464u;
    // packed zeros: weight-side data fetched a chunk of kPf groups ahead, so a
    // load has kPf groups of time to land before its group starts
    auto zero_word = [&](int gi) -> uint32_t {
      return (HAS_Z && n < N && gi < ng) ? static_cast<uint32_t>(a.qzeros[size_t(g0 + gi) * (N / 8) + n / 8]) : 0u;
    };
    uint32_t zcur[kPf], znxt[kPf];
    if (HAS_Z) {
#pragma unroll
      for (int j = 0; j < kPf; ++j) {
        zcur[j] = zero_word(j);
        znxt[j] = zero_word(kPf + j);
      }
    }
    uint32_t zbias = 0;
    for (int i = 0; i < nst; ++i) {
      const int s = i % kNS, ab = i % kNA;
      if (i % spg == 0) {
        const int gi = i / spg;
        int z = 8;
        if (HAS_Z) {
          if (gi % kPf == 0 && gi > 0) {
#pragma unroll
            for (int j = 0; j < kPf; ++j) {
              zcur[j] = znxt[j];
              znxt[j] = zero_word(gi + kPf + j);
            }
          }
          if (n < N) z = (zcur[gi % kPf] >> (4 * (n % 8))) & 15;
        }
        // 16-bit pair of (128 + z) in bf16 or (1024 + z) in fp16
        const uint32_t h = ACT_BF16 ? (0x4300u | uint32_t(z)) : (0x6400u | uint32_t(z));
        zbias = h | (h << 16);
      }
      // warp-uniform decisions: the warp synchronises before its arrival below
      if (!__all_sync(0xffffffffu, mbar_wait_sleep(&full[s], (i / kNS) & 1))) { *failed = 1; break; }
      if (i >= kNA && !__all_sync(0xffffffffu, mbar_wait_sleep(&a_empty[ab], ((i / kNA) - 1) & 1))) { *failed = 1; break; }
      const uint32_t* wrow = reinterpret_cast<const uint32_t*>(sW + size_t(s) * kPackedStageBytes) + col;
      tc_fence_after();
      uint32_t h[kACols];
#pragma unroll
      for (int r = 0; r < KS / 8; ++r) {
        const uint32_t w = wrow[r * kBN];
        const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
        const uint32_t c0123 = prmt(lo, hi, 0x5140u), c4567 = prmt(lo, hi, 0x7362u);
        h[4 * r + 0] = sub2<ACT_BF16>(prmt(c0123, magic, 0x4140u), zbias);
        h[4 * r + 1] = sub2<ACT_BF16>(prmt(c0123, magic, 0x4342u), zbias);
        h[4 * r + 2] = sub2<ACT_BF16>(prmt(c4567, magic, 0x4140u), zbias);
        h[4 * r + 3] = sub2<ACT_BF16>(prmt(c4567, magic, 0x4342u), zbias);
      }
      // this warp's lane quarter (columns 32 w ..) of the A stage
      const uint32_t taddr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + Tmem<MP, KS>::kA + ab * kACols;
#pragma unroll
      for (int c = 0; c < int(kACols); c += 32) tmem_st32(taddr + c, h + c);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&a_full[ab]);
    }
    pdl_wait();
  } else {
    // ------------------------------------------------------------ epilogue --
    const int col = threadIdx.x - 4 * 32;  // 0..127 == tensor-memory lane
    const int n = n0 + col;
    const uint16_t* SC = static_cast<const uint16_t*>(a.scales);
    // group scales: weight-side data, read before the dependency wait and then a
    // chunk of kPf groups ahead of their use (the loads come from HBM)
    auto scale_bits = [&](int gi) -> uint32_t {
      return (n < N && gi < ng) ? static_cast<uint32_t>(SC[size_t(g0 + gi) * N + n]) : 0u;
    };
    uint32_t cur[kPf], nxt[kPf];
#pragma unroll
    for (int j = 0; j < kPf; ++j) cur[j] = scale_bits(j);
    pdl_wait();
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    bool stop = false;
    for (int gb = 0; gb < ng && !stop; gb += kPf) {
#pragma unroll
      for (int j = 0; j < kPf; ++j) nxt[j] = scale_bits(gb + kPf + j);
#pragma unroll
      for (int j = 0; j < kPf; ++j) {
        const int gi = gb + j;
        if (gi >= ng) break;
        const int tb = gi & 1;
        const float sc = ACT_BF16 ? bf16_bits_to_f32(cur[j]) : f16_bits_to_f32(cur[j]);
        if (!__all_sync(0xffffffffu, mbar_wait_sleep(&t_full[tb], (gi / 2) & 1))) {
          *failed = 1;
          stop = true;
          break;
        }
        tc_fence_after();
        float d[MP];
#pragma unroll
        for (int c = 0; c < MP; c += 16) tmem_ld16(lane_addr + tb * MP + c, d + c);
        tc_fence_before();
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&t_empty[tb]);
#pragma unroll
        for (int m = 0; m < MP; ++m) acc[m] = fmaf(sc, d[m], acc[m]);
      }
#pragma unroll
      for (int j = 0; j < kPf; ++j) cur[j] = nxt[j];
    }
#pragma unroll
    for (int m = 0; m < MP; ++m) part[m * kBN + col] = acc[m];
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMMA) tmem_dealloc(tmem, kTmemCols);

  uint16_t* Y = static_cast<uint16_t*>(a.y);
  finish_tile<MP, kBN>(part, S, [&](int m, int c, float v) {
    const int nn = n0 + c;
    if (m < M && nn < N) Y[size_t(m) * N + nn] = f32_to_act<ACT_BF16>(v);
  });
}

template <int MP, int ACT, bool HZ, int KS>
cudaError_t launch_mma(const CUtensorMap& wmap, const CUtensorMap& xmap, const MmaArgs& a, int T, int S,
                       unsigned flags, cudaStream_t stream) {
  const void* kern = reinterpret_cast<const void*>(wq4_mma_kernel<MP, ACT, HZ, KS>);
  const size_t smem = SmemMma(MP, KS).total;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, T, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (S > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = S;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  if (flags & WQ_FLAG_PDL) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  void* args[3] = {const_cast<CUtensorMap*>(&wmap), const_cast<CUtensorMap*>(&xmap), const_cast<MmaArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, kern, args);
}

template <int MP, int KS>
cudaError_t dispatch_mp(const CUtensorMap& wmap, const CUtensorMap& xmap, const MmaArgs& a, int T, int S,
                        int act_bf16, bool has_z, unsigned flags, cudaStream_t stream) {
  if (act_bf16) return has_z ? launch_mma<MP, 1, true, KS>(wmap, xmap, a, T, S, flags, stream)
                             : launch_mma<MP, 1, false, KS>(wmap, xmap, a, T, S, flags, stream);
  return has_z ? launch_mma<MP, 0, true, KS>(wmap, xmap, a, T, S, flags, stream)
               : launch_mma<MP, 0, false, KS>(wmap, xmap, a, T, S, flags, stream);
}
template <int MP>
cudaError_t dispatch_ks(int KS, const CUtensorMap& wmap, const CUtensorMap& xmap, const MmaArgs& a, int T, int S,
                        int act_bf16, bool has_z, unsigned flags, cudaStream_t stream) {
  return KS == 128 ? dispatch_mp<MP, 128>(wmap, xmap, a, T, S, act_bf16, has_z, flags, stream)
                   : dispatch_mp<MP, 64>(wmap, xmap, a, T, S, act_bf16, has_z, flags, stream);
}

}  // namespace

cudaError_t launch_wq4_mma(const void* x, const int32_t* qweight, const void* scales, const int32_t* qzeros,
                           void* y, int M, int K, int N, int group, int act_bf16, unsigned flags,
                           cudaStream_t stream) {
  if (group % kBoxK != 0) return cudaErrorNotSupported;
  const int KS = group % 128 == 0 ? 128 : 64;  // one or more whole stages per scale group
  const int T = (N + kBN - 1) / kBN, units = K / group;
  const int sms = std::max(1, device_sm_count());
  int S = std::max(1, std::min(8, (sms + T / 2) / T));
  S = std::min(S, units);
  CUtensorMap wmap;
  if (!encode_tensor_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, qweight, N, K / 8, size_t(N) * 4, kBN, KS / 8,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  for (int m0 = 0; m0 < M; m0 += 64) {
    const int mc = std::min(64, M - m0);
    const int MP = mc <= 16 ? 16 : (mc <= 32 ? 32 : 64);
    if (SmemMma(MP, KS).total > static_cast<size_t>(device_max_smem())) return cudaErrorNotSupported;
    CUtensorMap xmap;
    const uint16_t* xc = static_cast<const uint16_t*>(x) + size_t(m0) * K;
    if (!encode_tensor_map_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, xc, K, mc, size_t(K) * 2, kBoxK, MP,
                              CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    MmaArgs args{static_cast<uint16_t*>(y) + size_t(m0) * N, scales, qzeros, mc, K, N, group};
    cudaError_t e;
    switch (MP) {
      case 16: e = dispatch_ks<16>(KS, wmap, xmap, args, T, S, act_bf16, qzeros != nullptr, flags, stream); break;
      case 32: e = dispatch_ks<32>(KS, wmap, xmap, args, T, S, act_bf16, qzeros != nullptr, flags, stream); break;
      default: e = dispatch_ks<64>(KS, wmap, xmap, args, T, S, act_bf16, qzeros != nullptr, flags, stream); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace wq
