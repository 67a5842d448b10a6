// wq_gemv4m.cu -- 4-bit weight-only GEMV / skinny GEMM (M <= 8) on the warp-level
// tensor-core MMA (mma.sync m16n8k16, fp32 accumulate).
//
// Definition ("Quantization CUDA", Int4 Weight Only Quantization / Weight Store
// and 量化粒度; act-order: "GPTQ算法解析", 4.1):
//   y[m,n] = sum_k x[m,k] * s[g(k),n] * (q[k,n] - z[g(k),n]).
// Storage: qweight int32 [K/8, N], nibble j of word [r, n] = code of row 8r+j.
//
// Why a tensor-core MMA for a memory-bound product: with one or a few rows of x
// the fused multiply-adds on the CUDA cores cost one instruction per weight and
// row of x; the MMA takes the product off the arithmetic pipes (all M <= 8 rows
// in one instruction), so each weight costs only its exact conversion:
//   * a LOP3 puts two nibbles into the mantissas of an fp16 (bf16) pair holding
//     1024 + q (128 + q), and one HSUB2 (or, for the nibbles read in place at
//     bit 4, one HFMA2 by 1/16) leaves q - z exactly: every value is a small
//     integer, so A is exact and so are the products with x in fp32;
//   * the group scale multiplies the fp32 accumulator once per 64 values of k.
//
// Fragment layout.  A = W^T tile (16 columns n x 16 values k), B = x^T (16 k x
// 8 rows m).  The order of k inside the MMA does not change the sum, so each
// thread takes whole 32-bit words: thread (g = lane/4, t = lane%4) reads, per
// 32 values of k, one 16-byte chunk = the words of columns 4g..4g+3 of one
// word row, and feeds its 8 nibbles to its own k slots of two m16 tiles
// (tile 0: columns 4g, 4g+1 as rows g, g+8; tile 1: columns 4g+2, 4g+3).  Its x
// values are the same 8 k of the same word row, taken from shared memory with
// one 16-byte load and paired by PRMT.
//
// Shared-memory banks.  Weights land through TMA boxes of 32 words x 32 word
// rows with the 128-byte swizzle (16-byte chunk c of row r stored at c ^ (r%8)).
// Thread t of a 64-k unit reads word rows 2t and 2t+1, so in every 8-lane phase
// of a 16-byte load the chunk indices g ^ 2t (g ^ (2t+1)) are all different.
//
// Work decomposition: as the CUDA-core kernels (column tiles of 128, split-K
// over a cluster of S CTAs, warp 8 the TMA producer), with 64-k units; warp w
// of the 8 consumers owns the 32-column slab w%4 and half w/4 of each stage.
#include "wq_gemv_common.cuh"
#include "wq_launch.h"

namespace wq {
namespace {

constexpr int kBN = 128;                               // columns per CTA tile
constexpr int kSlab = 32;                              // columns per swizzled box (one warp)
constexpr int kStageWR = 32;                           // packed word rows per stage
constexpr int kStageK = kStageWR * 8;                  // 256 values of k per stage
constexpr int kUnitWR = 8;                             // word rows per unit (64 values of k)
constexpr int kUnitK = kUnitWR * 8;
constexpr int kUnitsPerStage = kStageWR / kUnitWR;     // 4
constexpr int kBoxBytes = kStageWR * kSlab * 4;        // 4 KB
constexpr int kStageBytes = kBoxBytes * (kBN / kSlab);  // 16 KB
constexpr int kNS = 4;

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

// Split-K reduction for this fragment layout: the tile's 128 columns are
// split into S chunks (a multiple of 4 columns), chunk r owned by cluster rank
// r; the two warps of each slab in each of the S CTAs send one piece each.
struct TileReduceM {
  int S, chunk;
  __host__ __device__ TileReduceM(int S_) : S(S_), chunk(((kBN + S_ - 1) / S_ + 3) & ~3) {}
  __host__ __device__ int piece(int MT) const { return MT * chunk; }
  __host__ __device__ size_t recv_floats(int MT) const { return size_t(S) * 2 * piece(MT); }
  __host__ __device__ uint32_t recv_bytes(int MT, int owner) const {
    const int len = min(chunk, kBN - owner * chunk);
    return len > 0 ? uint32_t(S) * 2u * MT * len * 4u : 0u;
  }
};

struct Smem4M {
  size_t xst, xg, xfull, scl, zp, recv, bars, flag, total;
  __host__ __device__ Smem4M(int MT, int ng_max, int S, bool perm, int K) {
    size_t o = size_t(kNS) * kStageBytes;
    const size_t xstage = size_t(MT) * kStageK * 2 > size_t(kStageK) * 4 ? size_t(MT) * kStageK * 2 : size_t(kStageK) * 4;
    xst = o;   o = align16(o + kNS * xstage);
    xg = o;    o = align16(o + (perm ? size_t(kConsumerWarps) * MT * (kStageK / 2) * 2 : 0));
    xfull = o; o = align16(o + (perm ? size_t(MT) * K * 2 : 0));
    scl = o;   o = align16(o + size_t(ng_max) * kBN * 2);        // raw 16-bit scales
    zp = o;    o = align16(o + size_t(ng_max) * (kBN / 8) * 4);  // raw packed zeros
    recv = o;  o = align16(o + TileReduceM(S).recv_floats(MT) * 4);
    bars = o;  o = align16(o + size_t(2 * kNS + 1) * 8);
    flag = o;  o = align16(o + 16);
    total = o;
  }
  __host__ __device__ static size_t xstage_bytes(int MT) {
    return size_t(MT) * kStageK * 2 > size_t(kStageK) * 4 ? size_t(MT) * kStageK * 2 : size_t(kStageK) * 4;
  }
};

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return d;
}
__device__ __forceinline__ uint32_t hsub2_f16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hfma2_f16(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hsub2_bf16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// One packed word (8 codes of one column) -> four fp16/bf16 pairs of q - z:
// P[0] = codes (0, 4), P[1] = (1, 5), P[2] = (2, 6), P[3] = (3, 7) (low, high half).
// zsub = pair of (1024 + z) (fp16) or (128 + z) (bf16); zfma = pair of -(64 + z) (fp16).
template <int ACT_BF16>
__device__ __forceinline__ void convert_word(uint32_t w, uint32_t zsub, uint32_t zfma, uint32_t (&P)[4]) {
  if (ACT_BF16) {
    constexpr uint32_t kMagic = 0x43004300u;  // bf16 pair (128, 128)
    P[0] = hsub2_bf16(lop3_and_or(w, 0x000F000Fu, kMagic), zsub);
    P[1] = hsub2_bf16(lop3_and_or(w >> 4, 0x000F000Fu, kMagic), zsub);
    P[2] = hsub2_bf16(lop3_and_or(w >> 8, 0x000F000Fu, kMagic), zsub);
    P[3] = hsub2_bf16(lop3_and_or(w >> 12, 0x000F000Fu, kMagic), zsub);
  } else {
    constexpr uint32_t kMagic = 0x64006400u;    // fp16 pair (1024, 1024)
    constexpr uint32_t kSixteenth = 0x2C002C00u;  // fp16 pair (1/16, 1/16)
    const uint32_t w8 = w >> 8;
    P[0] = hsub2_f16(lop3_and_or(w, 0x000F000Fu, kMagic), zsub);
    P[1] = hfma2_f16(lop3_and_or(w, 0x00F000F0u, kMagic), kSixteenth, zfma);  // (1024 + 16q) / 16 - 64 - z
    P[2] = hsub2_f16(lop3_and_or(w8, 0x000F000Fu, kMagic), zsub);
    P[3] = hfma2_f16(lop3_and_or(w8, 0x00F000F0u, kMagic), kSixteenth, zfma);
  }
}

// Code pair `pi` (0: codes 0,4; 1: 1,5; 2: 2,6; 3: 3,7) of one packed word as q - z.
template <int ACT_BF16, int PI>
__device__ __forceinline__ uint32_t convert_pair(uint32_t w, uint32_t zsub, uint32_t zfma) {
  if (ACT_BF16) {
    return hsub2_bf16(lop3_and_or(w >> (4 * PI), 0x000F000Fu, 0x43004300u), zsub);
  } else {
    const uint32_t ws = (PI >= 2) ? (w >> 8) : w;
    if (PI & 1) return hfma2_f16(lop3_and_or(ws, 0x00F000F0u, 0x64006400u), 0x2C002C00u, zfma);
    return hsub2_f16(lop3_and_or(ws, 0x000F000Fu, 0x64006400u), zsub);
  }
}

template <int ACT_BF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  if (ACT_BF16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int ACT_BF16>
__device__ __forceinline__ float scale_to_f32(uint32_t bits16) {
  return ACT_BF16 ? bf16_bits_to_f32(bits16) : f16_bits_to_f32(bits16);
}

// MT = rows of x the instance handles (1, 2, 4 or 8: one MMA column block).
// PERM: rows of the weights were sorted by act-order group ahead of time
// (wq4_actorder_prepare); stage row i multiplies x[perm[i]], the whole x sits
// in shared memory and the "x" map streams the matching slice of perm.
template <int MT, int ACT_BF16, bool HAS_Z, bool PERM>
__global__ void __launch_bounds__(kGemvThreads, 1)
    k4m_gemv_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                    const GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int S = gridDim.x;
  const Smem4M L(MT, a.ng_max, S, PERM, a.K);
  const TileReduceM R(S);
  uint8_t* wst = smem;
  uint8_t* xst = smem + L.xst;
  const size_t xstage = Smem4M::xstage_bytes(MT);
  uint16_t* scl = reinterpret_cast<uint16_t*>(smem + L.scl);
  uint32_t* zp = reinterpret_cast<uint32_t*>(smem + L.zp);
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kNS;
  uint64_t* recv_bar = empty + kNS;
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L.flag);  // producer's
  volatile int* cfailed = failed + 1;                                       // consumers'

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.y * kBN;
  const int M = a.M, K = a.K, N = a.N, gsz = a.group;
  int u0, u1;
  split_range(K / kUnitK, S, blockIdx.x, u0, u1);
  const int n_loads = (u1 - u0 + kUnitsPerStage - 1) / kUnitsPerStage;
  const UnitGroups ug(gsz, kUnitK);
  const int g0 = ug.of(u0);
  const int ng = (u1 > u0) ? (kUnitK * u1 - 1) / gsz - g0 + 1 : 0;
  constexpr uint32_t kXBytes = PERM ? kStageK * 4 : MT * kStageK * 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *failed = 0;
    *cfailed = 0;
    if (S == 1) {
      mbar_init(recv_bar, kConsumerThreads);
    } else {
      mbar_init(recv_bar, 1);
      const uint32_t rb = R.recv_bytes(MT, cluster_rank());
      if (rb) mbar_expect_tx(recv_bar, rb);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (S > 1) cluster_arrive_relaxed();
  pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer
    int issued = 0;
    if (lane == 0 && n_loads > 0) {
      prefetch_tensormap(&wmap);
      prefetch_tensormap(&xmap);
      const uint64_t pol = l2_evict_first_policy();
      const int wr0 = kUnitWR * u0;
      const int pre = n_loads < kNS ? n_loads : kNS;
      for (int it = 0; it < pre; ++it) {
        mbar_expect_tx(&full[it], kStageBytes + kXBytes);
#pragma unroll
        for (int b = 0; b < kBN / kSlab; ++b)
          tma_load_2d(wst + size_t(it) * kStageBytes + b * kBoxBytes, &wmap, &full[it], n0 + b * kSlab,
                      wr0 + it * kStageWR, pol);
      }
      pdl_wait();
      for (int it = 0; it < pre; ++it)
        tma_load_2d(xst + size_t(it) * xstage, &xmap, &full[it], kUnitK * u0 + it * kStageK, 0, 0ull);
      issued = pre;
      for (int it = kNS; it < n_loads; ++it) {
        const int s = it % kNS;
        if (*failed || !mbar_wait(&empty[s], ((it / kNS) - 1) & 1)) {
          *failed = 1;
          break;
        }
        mbar_expect_tx(&full[s], kStageBytes + kXBytes);
#pragma unroll
        for (int b = 0; b < kBN / kSlab; ++b)
          tma_load_2d(wst + size_t(s) * kStageBytes + b * kBoxBytes, &wmap, &full[s], n0 + b * kSlab,
                      wr0 + it * kStageWR, pol);
        tma_load_2d(xst + size_t(s) * xstage, &xmap, &full[s], kUnitK * u0 + it * kStageK, 0, 0ull);
        ++issued;
      }
    }
    pdl_wait();
    if (lane == 0 && *failed) drain_stages<kNS>(full, issued);
    __syncwarp();
    if (S > 1) cluster_wait();
  } else {
    // --------------------------------------------------------------- consumers
    const int tid = threadIdx.x;
    // weight-side tables of this CTA's groups, read before the dependency wait:
    // scl[g][c] = raw 16-bit scale, zp[g][c/8] = raw packed zeros (8 per word)
    {
      const uint16_t* SC = static_cast<const uint16_t*>(a.scales);
      const int32_t* QZ = static_cast<const int32_t*>(a.zeros);
      for (int i = tid; i < ng * (kBN / 2); i += kConsumerThreads) {
        const int gr = i / (kBN / 2), c = 2 * (i % (kBN / 2));
        uint32_t v = 0;
        if (n0 + c < N) v = *reinterpret_cast<const uint32_t*>(SC + size_t(g0 + gr) * N + n0 + c);
        reinterpret_cast<uint32_t*>(scl)[i] = v;
      }
      for (int i = tid; i < ng * (kBN / 8); i += kConsumerThreads) {
        const int gr = i / (kBN / 8), c = i % (kBN / 8);
        zp[i] = (HAS_Z && n0 + 8 * c < N) ? static_cast<uint32_t>(QZ[size_t(g0 + gr) * (N / 8) + n0 / 8 + c])
                                          : 0x88888888u;
      }
    }
    pdl_wait();
    const uint16_t* xfull = reinterpret_cast<const uint16_t*>(smem + L.xfull);
    if (PERM) {  // the whole x in shared memory (rows >= M read as zero)
      uint4* xf = reinterpret_cast<uint4*>(smem + L.xfull);
      const int chunks_per_row = K / 8;
      for (int i = tid; i < MT * chunks_per_row; i += kConsumerThreads) {
        const int m = i / chunks_per_row, c = i % chunks_per_row;
        xf[i] = (m < M) ? reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + size_t(m) * K)[c]
                        : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    consumer_sync(kConsumerThreads);  // tables (and x) complete before any warp uses them

    const int g = lane >> 2, t = lane & 3;
    const int slab = warp & 3, khalf = warp >> 2;
    const int col4 = slab * kSlab + 4 * g;  // this thread's 4 columns within the tile
    uint16_t* xg = reinterpret_cast<uint16_t*>(smem + L.xg) + size_t(warp) * MT * (kStageK / 2);

    // acc: running sums (scale applied); tmp[set]: the current group's MMA sums,
    // two independent sets (even / odd word rows) so that two MMA chains overlap
    float acc[2][4], tmp[2][2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[j][i] = tmp[0][j][i] = tmp[1][j][i] = 0.f;
    int cur_g = -1;  // group held in tmp (-1: none)
    uint32_t zsv[4] = {0u, 0u, 0u, 0u}, zfv[4] = {0u, 0u, 0u, 0u};

    // acc += s(group) * (tmp[0] + tmp[1]); tmp = 0
    auto fold = [&](int gi) {
      const uint2 sb = *reinterpret_cast<const uint2*>(scl + gi * kBN + col4);
      const float sv[4] = {scale_to_f32<ACT_BF16>(sb.x & 0xFFFFu), scale_to_f32<ACT_BF16>(sb.x >> 16),
                           scale_to_f32<ACT_BF16>(sb.y & 0xFFFFu), scale_to_f32<ACT_BF16>(sb.y >> 16)};
#pragma unroll
      for (int tl = 0; tl < 2; ++tl)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[tl][i] = fmaf(sv[2 * tl + (i >> 1)], tmp[0][tl][i] + tmp[1][tl][i], acc[tl][i]);
          tmp[0][tl][i] = tmp[1][tl][i] = 0.f;
        }
    };

    for (int it = 0; it < n_loads; ++it) {
      const int s = it % kNS;
      if (!mbar_wait(&full[s], (it / kNS) & 1)) *cfailed = 1;
      if (*cfailed) break;
      const uint8_t* xs = xst + size_t(s) * xstage;
      if (PERM) {  // this warp's half-stage of x in sorted order: xg[m][kk]
        const int32_t* pv = reinterpret_cast<const int32_t*>(xs) + khalf * (kStageK / 2);
#pragma unroll
        for (int i = 0; i < (kStageK / 2) / 32; ++i) {
          const int kk = lane + 32 * i;
          int kp = pv[kk];
          kp = min(max(kp, 0), K - 1);  // out-of-range entries are clamped, never read out of bounds
#pragma unroll
          for (int m = 0; m < MT; ++m) xg[m * (kStageK / 2) + kk] = xfull[size_t(m) * K + kp];
        }
        __syncwarp();
      }
      const uint8_t* box = wst + size_t(s) * kStageBytes + slab * kBoxBytes;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int u = u0 + kUnitsPerStage * it + 2 * khalf + j;
        if (u >= u1) break;
        const int gi = ug.of(u) - g0;
        if (gi != cur_g) {  // a new scale group: apply the finished one, load the new zeros
          if (cur_g >= 0) fold(cur_g);
          cur_g = gi;
          // zero pairs of this thread's 4 columns, built from the nibbles:
          // fp16 1024 + z = 0x6400 | z, -(64 + z) = 0xD400 | z << 4; bf16 128 + z = 0x4300 | z
          const uint32_t zw = zp[gi * (kBN / 8) + col4 / 8] >> (4 * (col4 % 8));
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t z = (zw >> (4 * c)) & 15u;
            const uint32_t hs = ACT_BF16 ? (0x4300u | z) : (0x6400u | z);
            const uint32_t hf = 0xD400u | (z << 4);
            zsv[c] = hs | (hs << 16);
            zfv[c] = hf | (hf << 16);
          }
        }
        const int rb = kUnitWR * (2 * khalf + j);  // first word row of the unit within the stage
        uint4 wv[2], xv[2];
#pragma unroll
        for (int ab = 0; ab < 2; ++ab) {
          const int r = rb + 2 * t + ab;  // this thread's word rows
          wv[ab] = lds128(smem_u32(box + r * 128 + (((g ^ (r & 7)) & 7) << 4)));
          xv[ab] = make_uint4(0u, 0u, 0u, 0u);
          if (g < MT) {
            if (PERM)
              xv[ab] = lds128(smem_u32(xg + g * (kStageK / 2) + 8 * (r - 16 * khalf)));
            else
              xv[ab] = lds128(smem_u32(xs + (size_t(g) * kStageK + 8 * r) * 2));
          }
        }
#pragma unroll
        for (int ab = 0; ab < 2; ++ab) {
          const uint32_t w4[4] = {wv[ab].x, wv[ab].y, wv[ab].z, wv[ab].w};
          const uint32_t b[4] = {prmt(xv[ab].x, xv[ab].z, 0x5410u),   // (x0, x4)
                                 prmt(xv[ab].x, xv[ab].z, 0x7632u),   // (x1, x5)
                                 prmt(xv[ab].y, xv[ab].w, 0x5410u),   // (x2, x6)
                                 prmt(xv[ab].y, xv[ab].w, 0x7632u)};  // (x3, x7)
#pragma unroll
          for (int tl = 0; tl < 2; ++tl) {
            // operands in MMA order: rows g (word 2tl) and g+8 (word 2tl+1), low then high k slots
            const uint32_t we = w4[2 * tl], wo = w4[2 * tl + 1];
            const uint32_t zse = zsv[2 * tl], zso = zsv[2 * tl + 1], zfe = zfv[2 * tl], zfo = zfv[2 * tl + 1];
            mma_16816<ACT_BF16>(tmp[ab][tl], convert_pair<ACT_BF16, 0>(we, zse, zfe), convert_pair<ACT_BF16, 0>(wo, zso, zfo),
                                convert_pair<ACT_BF16, 1>(we, zse, zfe), convert_pair<ACT_BF16, 1>(wo, zso, zfo), b[0], b[1]);
            mma_16816<ACT_BF16>(tmp[ab][tl], convert_pair<ACT_BF16, 2>(we, zse, zfe), convert_pair<ACT_BF16, 2>(wo, zso, zfo),
                                convert_pair<ACT_BF16, 3>(we, zse, zfe), convert_pair<ACT_BF16, 3>(wo, zso, zfo), b[2], b[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (cur_g >= 0) fold(cur_g);

    // ------------------------------------------------ split-K partial sums out
    // this thread holds rows m = 2t, 2t+1 of columns col4 .. col4 + 3
    const int col = col4, r_own = col / R.chunk, cc = col % R.chunk;
    if (S == 1) {
      float* slot = recv + size_t(khalf) * R.piece(MT);
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int m = 2 * t + p;
        if (m < MT)
          *reinterpret_cast<float4*>(slot + m * R.chunk + cc) =
              make_float4(acc[0][p], acc[0][2 + p], acc[1][p], acc[1][2 + p]);
      }
      mbar_arrive(recv_bar);  // release: the stores above are visible to the waiter
    } else {
      __syncwarp();
      cluster_wait();
      const uint32_t me = cluster_rank();
      float* slot = recv + (size_t(me) * 2 + khalf) * R.piece(MT);
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int m = 2 * t + p;
        if (m < MT)
          st_async_v4_to_rank(smem_u32(slot + m * R.chunk + cc), acc[0][p], acc[0][2 + p], acc[1][p], acc[1][2 + p],
                              smem_u32(recv_bar), uint32_t(r_own));
      }
    }
  }

  // ------------------------------------------ owner: sum the pieces, store y
  {
    const uint32_t me = S > 1 ? cluster_rank() : 0u;
    const int c0 = int(me) * R.chunk;
    const int len = min(R.chunk, kBN - c0);
    if (len > 0 && mbar_wait(recv_bar, 0)) {
      uint16_t* Y = static_cast<uint16_t*>(a.y);
      const int n_pieces = S * 2;
      for (int e = threadIdx.x; e < MT * len; e += blockDim.x) {
        const int m = e / len, c = e % len, n = n0 + c0 + c;
        float v = 0.f;
        for (int q = 0; q < n_pieces; ++q) v += recv[size_t(q) * R.piece(MT) + m * R.chunk + c];
        if (m < M && n < N) Y[size_t(m) * N + n] = f32_to_act<ACT_BF16>(v);
      }
    }
  }
}

template <int MT, int ACT, bool HZ, bool PERM>
cudaError_t launch_m(const LaunchPlan& p, const CUtensorMap& w, const CUtensorMap& x, const GemvArgs& a) {
  const CUtensorMap* maps[2] = {&w, &x};
  return launch_gemv_kernel(reinterpret_cast<const void*>(k4m_gemv_kernel<MT, ACT, HZ, PERM>), p,
                            Smem4M(MT, a.ng_max, p.S, PERM, a.K).total, maps, 2, a);
}

template <int MT>
cudaError_t dispatch_m(const LaunchPlan& p, const CUtensorMap& w, const CUtensorMap& x, const GemvArgs& a,
                       int act_bf16, bool has_z, bool perm) {
  if (perm) {
    if (act_bf16) return has_z ? launch_m<MT, 1, true, true>(p, w, x, a) : launch_m<MT, 1, false, true>(p, w, x, a);
    return has_z ? launch_m<MT, 0, true, true>(p, w, x, a) : launch_m<MT, 0, false, true>(p, w, x, a);
  }
  if (act_bf16) return has_z ? launch_m<MT, 1, true, false>(p, w, x, a) : launch_m<MT, 1, false, false>(p, w, x, a);
  return has_z ? launch_m<MT, 0, true, false>(p, w, x, a) : launch_m<MT, 0, false, false>(p, w, x, a);
}

}  // namespace

int wq4m_unit_k() { return kUnitK; }
int wq4m_stage_k() { return kStageK; }

size_t wq4m_gemv_smem_bytes(int MT, int ng_max, int S, bool perm, int K) {
  return Smem4M(MT, ng_max, S, perm, K).total;
}

cudaError_t launch_wq4m_gemv(const LaunchPlan& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                             const GemvArgs& a, int act_bf16, bool has_z, bool perm) {
  switch (p.MT) {
    case 1: return dispatch_m<1>(p, wmap, xmap, a, act_bf16, has_z, perm);
    case 2: return dispatch_m<2>(p, wmap, xmap, a, act_bf16, has_z, perm);
    case 4: return dispatch_m<4>(p, wmap, xmap, a, act_bf16, has_z, perm);
    case 8: return dispatch_m<8>(p, wmap, xmap, a, act_bf16, has_z, perm);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace wq
