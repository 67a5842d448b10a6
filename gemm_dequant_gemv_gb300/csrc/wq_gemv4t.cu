// wq_gemv4t.cu -- 4-bit weight-only GEMV / skinny GEMM (M <= 32) on the
// warp-level tensor-core MMA (mma.sync m16n8k16, fp32 accumulate).
//
// Definition ("Quantization CUDA", Int4 Weight Only Quantization / Weight Store
// and 量化粒度; act-order: "GPTQ算法解析", 4.1 内存-计算权衡):
//   y[m,n] = sum_k x[m,k] * s[g(k),n] * (q[k,n] - z[g(k),n]).
//
// Why the MMA for a memory-bound product: every weight code must be converted
// and multiplied once per row of x.  On GB300 the integer / logic pipe (LOP3,
// PRMT, shifts) and the packed half-precision pipe run at half the rate of the
// fp32 FMA pipe, and packed fp32 FMAs contend with the logic pipe, so the
// CUDA-core form (one PRMT and half a packed FMA per code) issues at well
// under half of the SM's rate.  Here each code costs only its exact conversion
// (5/8 of a logic op and 1/2 of a packed half op); the products of up to 8
// rows of x come from one MMA per 256 codes, and 9 - 32 rows from two or
// four (n-tiles of 8 rows) that share the converted A fragments:
//   * one LOP3 puts two nibbles into the mantissas of an fp16 (bf16) pair
//     holding 1024 + q (128 + q), and one HSUB2 (or, for nibbles read in place
//     at bit 4, one HFMA2 by 1/16) leaves q - z exactly: A is exact, and so are
//     the products with x in the fp32 accumulator;
//   * the group scale multiplies the fp32 accumulators once per group.
//
// Fragments.  A = the weight tile (16 columns n x 16 values k), B = x^T (16 k
// x 8 rows m).  The order of k inside one MMA does not change the sum, so each
// thread (g = lane/4, t = lane%4) takes whole 32-bit words: per 64-value unit
// (8 word rows), word rows 2t and 2t+1 of columns 4g .. 4g+3 of the warp's
// 32-column slab, two 16-byte loads.  Columns 4g, 4g+1 are rows g, g+8 of MMA
// tile 0, columns 4g+2, 4g+3 those of tile 1; nibbles (j, j+4) of a word
// fill the thread's k slots of one MMA half, and its x values are the same
// eight k of the same word row, paired by PRMT.
//
// Weight layouts, both read conflict-free:
//   * GPTQ [K/8, N]: per stage and slab one 2D TMA box of 32 words x 64 word
//     rows with the 128-byte swizzle (16-byte chunk c of row r at c ^ (r%8));
//     thread t's rows 2t, 2t+1 put the 8 lanes of every load phase on 8
//     different chunks.  The slabs' boxes are issued by one producer lane
//     each; the whole GPTQ matrix streams through such boxes at ~5.6 TB/s on
//     GB300 when nothing is computed (measured), faster than per-thread
//     16-byte loads or cp.async of the same words.
//   * tiled (wq4_repack_tiled): the same words reordered once so that each
//     1 KB block (one 64-value unit of one slab) is contiguous, each thread's
//     16 bytes sit at lane * 16, and the blocks of one unit follow each other
//     over the slabs: a CTA's columns of one unit are one 1D bulk copy and
//     the loads are conflict-free without swizzle.
//
// Work decomposition: a CTA owns a tile of nslab slabs (32 * nslab columns)
// and a K-slice; the S CTAs of a cluster split K and add their partial sums
// through distributed shared memory.  nslab and S are chosen per shape so
// that the whole grid is resident at once (about one CTA per SM).  Two
// consumer warps per slab split each 512-value stage; the last warp is the
// producer.  x is staged per stage by TMA next to the weights (all M rows;
// with several n-tiles the rows past M are the box's zero fill).  Without a
// cluster the partial sums reuse the weight ring once every consumer is done.
// PERM (rows sorted by act-order group once ahead of time): sorted row i
// multiplies x[perm[i]]; each CTA gathers x of its K-slice through perm into
// shared memory once, right after the dependency wait.
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/wq.h"
#include "wq_gemv_common.cuh"
#include "wq_launch.h"

namespace wq {

namespace {

constexpr int kSlabCols = 32;
constexpr int kUnitK = 64;                               // 8 word rows
constexpr int kUnitBytes = kSlabCols * (kUnitK / 8) * 4;  // 1 KB
constexpr int kStageUnits = 8;
constexpr int kStageK = kStageUnits * kUnitK;            // 512
constexpr int kSlabStageBytes = kStageUnits * kUnitBytes;  // 8 KB
constexpr int kKW = 2;                                   // consumer warps per slab (x staged per stage)
constexpr int kKWPerm = 4;                               // consumer warps per slab (act-order, gathered x)
__host__ __device__ constexpr int kw_of(bool perm) { return perm ? kKWPerm : kKW; }
constexpr int kWarpK = kStageUnits / kKW * kUnitK;       // 256 values of k per warp and stage
static_assert(kWarpK == 256 && kStageK == 512, "one 256-value TMA box of x per consumer warp's half of a stage");

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }
__host__ __device__ inline size_t align1k(size_t v) { return (v + 1023) & ~size_t(1023); }
__host__ __device__ inline size_t align128(size_t v) { return (v + 127) & ~size_t(127); }

struct Smem4T {
  size_t ring, xst, xg, pv, scl, zp, recv, bars, flag, total;
  // krange: values of k of the largest K-slice (the gathered x of the act-order path)
  __host__ __device__ Smem4T(int nslab, int NS, int MT, int S, int ng_max, bool perm, int krange) {
    const int nown = (nslab + S - 1) / S;
    size_t o = 0;
    ring = o;  o = align1k(o + size_t(NS) * nslab * kSlabStageBytes);
    xst = o;   o = align16(o + (perm ? 0 : size_t(NS) * xstage_bytes(MT)));
    xg = o;    o = align16(o + (perm ? size_t(MT + 1) * krange * 2 : 0));
    pv = o;    o = align128(o + (perm ? size_t(krange) * 4 : 0));
    scl = o;   o = align128(o + size_t(ng_max) * nslab * kSlabCols * 2);    // TMA destinations: 128-byte aligned
    zp = o;    o = align16(o + size_t(ng_max) * nslab * (kSlabCols / 8) * 4);
    // the partial sums: without a cluster (S == 1) they reuse the ring, which
    // every consumer has finished with by then (it holds at least two stages:
    // nslab * 16 KB >= the KW * nslab * MT * 128 bytes of pieces for MT <= 32)
    if (S == 1) {
      recv = ring;
    } else {
      recv = o;  o = align16(o + size_t(S) * kw_of(perm) * nown * MT * kSlabCols * 4);
    }
    bars = o;  o = align16(o + size_t(2 * NS + 3) * 8);
    flag = o;  o = align16(o + 16);
    total = o;
  }
  // x stage: per 256-value half, MT rows of the stage's x and one zero row
  // (the B operand of lanes whose row is >= MT)
  __host__ __device__ static size_t xstage_bytes(int MT) { return size_t(MT + 1) * kStageK * 2; }
};

struct Args4T {
  const void* x;
  void* y;
  const void* scales;
  const int32_t* qzeros;   // null: symmetric zero 8
  const uint8_t* wtiled;   // tiled weights (tiled layout only)
  const int32_t* perm;     // act-order sort (PERM only)
  int M, K, N, group;
  int MT, nslab, NS, ng_max;
  int gshift;              // log2(units per group)
  int krange;              // values of k of the largest K-slice (multiple of 64)
  int tma_tables;          // scales (and zeros) of the CTA's groups by one TMA box each
};

__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<const __half2*>(&u); }
__device__ __forceinline__ __nv_bfloat162 as_b2(uint32_t u) { return *reinterpret_cast<const __nv_bfloat162*>(&u); }
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }
__device__ __forceinline__ uint32_t b2_bits(__nv_bfloat162 h) { return *reinterpret_cast<const uint32_t*>(&h); }

// Code pair PI of a packed word as q - z: PI = 0: codes (0, 4), 1: (1, 5),
// 2: (2, 6), 3: (3, 7) in the (low, high) halves.  zsub = pair of -(1024 + z)
// (fp16) or -(128 + z) (bf16); zfma = pair of -(64 + z) (fp16 only).  The
// subtraction is a packed FMA (the floating-point pipe, beside the logic ops).
template <int ACT_BF16, int PI>
__device__ __forceinline__ uint32_t convert_pair(uint32_t w, uint32_t w8, uint32_t zsub, uint32_t zfma) {
  if (ACT_BF16) {
    const uint32_t v = lop3_and_or(PI == 0 ? w : (w >> (4 * PI)), 0x000F000Fu, 0x43004300u);
    return b2_bits(__hfma2(as_b2(v), as_b2(0x3F803F80u), as_b2(zsub)));
  } else {
    const uint32_t ws = (PI >= 2) ? w8 : w;
    if (PI & 1) {  // (1024 + 16 q) / 16 - 64 - z
      const uint32_t v = lop3_and_or(ws, 0x00F000F0u, 0x64006400u);
      return h2_bits(__hfma2(as_h2(v), as_h2(0x2C002C00u), as_h2(zfma)));
    }
    const uint32_t v = lop3_and_or(ws, 0x000F000Fu, 0x64006400u);
    return h2_bits(__hfma2(as_h2(v), as_h2(0x3C003C00u), as_h2(zsub)));
  }
}

template <int ACT_BF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  if (ACT_BF16)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 1D bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}


// Act-order instances (short K-slices, chained in a decode step) run four
// consumer warps per slab: more warps in flight for the latency of the
// conversion and MMA chains of a short slice.
constexpr int kMaxSlabsPerm = 5;
// NT: 8-row n-tiles of the MMA (rows of x: NT = 1 up to 8, 2 up to 16, 4 up
// to 32); the converted A fragments serve every n-tile.
template <int ACT_BF16, bool HAS_Z, bool PERM, bool TILED, int NT>
__global__ void __launch_bounds__(PERM ? (kMaxSlabsPerm * kKWPerm + 1) * 32 : (NT == 4 ? 13 : 17) * 32, 1)
    k4t_gemv_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap wmap8,
                    const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap smap,
                    const __grid_constant__ CUtensorMap zmap, const Args4T a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int S = gridDim.x;
  const int nslab = a.nslab, NS = a.NS, MT = a.MT;
  constexpr int KW = kw_of(PERM), UPW = kStageUnits / KW;  // warps per slab, units per warp and stage
  const int W = nslab * KW;  // consumer warps
  const Smem4T L(nslab, NS, MT, S, a.ng_max, PERM, a.krange);
  uint8_t* ring = smem + L.ring;
  uint8_t* xst = smem + L.xst;
  const size_t xstage = Smem4T::xstage_bytes(MT);
  const size_t stage_w = size_t(nslab) * kSlabStageBytes;
  uint16_t* xg = reinterpret_cast<uint16_t*>(smem + L.xg);
  uint16_t* scl = reinterpret_cast<uint16_t*>(smem + L.scl);
  uint32_t* zp = reinterpret_cast<uint32_t*>(smem + L.zp);
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + NS;
  uint64_t* recv_bar = empty + NS;
  uint64_t* pbar = recv_bar + 1;  // the perm slice (act-order)
  uint64_t* tbar = pbar + 1;      // the scale and zero tables
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L.flag);  // producer's
  volatile int* cfailed = failed + 1;                                       // consumers'

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = a.M, K = a.K, N = a.N, gsz = a.group;
  const int BN = nslab * kSlabCols;
  const int n0 = blockIdx.y * BN;
  const int units = K / kUnitK;
  int u0, u1;
  split_range(units, S, blockIdx.x, u0, u1);
  const int n_stages = (u1 - u0 + kStageUnits - 1) / kStageUnits;
  const uint32_t rank = S > 1 ? cluster_rank() : 0u;
  const int nown_max = (nslab + S - 1) / S;
  const int nown = int(rank) < nslab ? (nslab - int(rank) + S - 1) / S : 0;
  const int g0 = (kUnitK * u0) / gsz;
  const int ng = (u1 > u0) ? (kUnitK * u1 - 1) / gsz - g0 + 1 : 0;
  // tiled layout: slabs of the matrix that exist (N is a multiple of 32 there)
  const int slab0 = n0 / kSlabCols;
  const int nvalid = TILED ? max(0, min(nslab, N / kSlabCols - slab0)) : nslab;
  const int krp = a.krange;  // row pitch of the gathered x (values)

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], W);
    }
    mbar_init(pbar, 1);
    mbar_init(tbar, 1);
    *failed = 0;
    *cfailed = 0;
    if (S == 1) {
      mbar_init(recv_bar, W * 32);
    } else {
      mbar_init(recv_bar, 1);
      const uint32_t rb = uint32_t(S) * KW * nown * MT * kSlabCols * 4;
      if (rb) mbar_expect_tx(recv_bar, rb);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (S > 1) cluster_arrive_relaxed();
  pdl_launch_dependents();

  if (warp == W) {
    // ------------------------------------------------------------------ producer
    // GPTQ layout: lane l < nslab issues slab l's box of every stage; tiled
    // layout: lane u < 8 issues unit u's copy (the CTA's slabs of one unit are
    // contiguous).  Lane 0 owns the barriers and the x copies.
    int issued = 0;
    auto stage_units = [&](int it) { return min(kStageUnits, u1 - u0 - kStageUnits * it); };
    auto stage_bytes = [&](int it) -> uint32_t {
      const int nu = stage_units(it);
      const uint32_t wb = uint32_t(TILED ? nvalid : nslab) * nu * kUnitBytes;
      return wb + (PERM ? 0u : uint32_t(MT) * kStageK * 2);
    };
    // x of stage it: boxes of 256 values (the TMA limit per dimension), box h at
    // rows [h][0 .. MT) of the stage's [2][MT + 1][256] layout
    auto issue_x = [&](int it, int s) {
      for (int h = 0; h < kStageK / 256; ++h)
        tma_load_2d(xst + size_t(s) * xstage + h * (MT + 1) * 256 * 2, &xmap, &full[s],
                    kUnitK * u0 + kStageK * it + 256 * h, 0, 0ull);
    };
    auto issue_weights = [&](int it, int s) {
      const int nu = stage_units(it);
      const int ustart = u0 + kStageUnits * it;
      if (TILED) {
        if (lane < nu && nvalid > 0)
          bulk_load(ring + size_t(s) * stage_w + size_t(lane) * nslab * kUnitBytes,
                    a.wtiled + (size_t(ustart + lane) * (N / kSlabCols) + slab0) * kUnitBytes,
                    uint32_t(nvalid) * kUnitBytes, &full[s]);
        return;
      }
      if (lane >= nslab) return;
      uint8_t* dst = ring + size_t(s) * stage_w + size_t(lane) * kSlabStageBytes;
      if (nu == kStageUnits) {
        tma_load_2d(dst, &wmap, &full[s], n0 + lane * kSlabCols, 8 * ustart, l2_evict_first_policy());
      } else {
        for (int i = 0; i < nu; ++i)
          tma_load_2d(dst + i * kUnitBytes, &wmap8, &full[s], n0 + lane * kSlabCols, 8 * (ustart + i),
                      l2_evict_first_policy());
      }
    };
    const uint32_t tbytes = uint32_t(a.ng_max) * BN * 2 + (HAS_Z ? uint32_t(a.ng_max) * (BN / 8) * 4 : 0u);
    if (a.tma_tables && lane == 0 && u1 > u0) {  // this CTA's scale (and zero) rows: one box each
      mbar_expect_tx(tbar, tbytes);
      tma_load_2d(scl, &smap, tbar, n0, g0, 0ull);
      if (HAS_Z) tma_load_2d(zp, &zmap, tbar, n0 / 8, g0, 0ull);
    }
    if (PERM && lane == 0 && u1 > u0) {  // the perm slice is weight-side data: before the dependency wait
      mbar_expect_tx(pbar, uint32_t(u1 - u0) * kUnitK * 4);
      bulk_load(smem + L.pv, a.perm + kUnitK * u0, uint32_t(u1 - u0) * kUnitK * 4, pbar);
    }
    if (n_stages > 0) {
      if (lane == 0) {
        if (!TILED) {
          prefetch_tensormap(&wmap);
          prefetch_tensormap(&wmap8);
        }
        if (!PERM) prefetch_tensormap(&xmap);
      }
      const int pre = n_stages < NS ? n_stages : NS;
      for (int it = 0; it < pre; ++it) {
        if (lane == 0) mbar_expect_tx(&full[it], stage_bytes(it));
        __syncwarp();
        issue_weights(it, it);
      }
      pdl_wait();
      if (!PERM && lane == 0)
        for (int it = 0; it < pre; ++it) issue_x(it, it);
      issued = pre;
      int s = 0;
      uint32_t ph = 0;  // parity of the empty phase awaited in slot s
      for (int it = NS; it < n_stages; ++it) {
        if (lane == 0) {
          if (*failed || !mbar_wait_sleep(&empty[s], ph)) *failed = 1;
          else mbar_expect_tx(&full[s], stage_bytes(it));
        }
        __syncwarp();
        if (*failed) break;
        issue_weights(it, s);
        if (!PERM && lane == 0) issue_x(it, s);
        ++issued;
        if (++s == NS) {
          s = 0;
          ph ^= 1u;
        }
      }
    } else {
      pdl_wait();
    }
    if (lane == 0 && *failed) {
      drain_stages_rt(full, NS, issued);
      if (PERM && u1 > u0) mbar_wait(pbar, 0);  // the copies land before the shared memory goes away
      if (a.tma_tables && u1 > u0) mbar_wait(tbar, 0);
    }
    __syncwarp();
    if (S > 1) cluster_wait();
  } else {
    // ----------------------------------------------------------------- consumers
    const int tid = threadIdx.x;
    const int nthr = W * 32;
    // weight-side tables of this CTA's groups: scl[g][c] = raw 16-bit scale,
    // zp[g][c/8] = raw packed zeros (8 per word).  Normally one TMA box each,
    // issued by the producer at the start; where the zeros' row pitch rules a
    // box out, read here before the dependency wait, four loads in flight per
    // thread (a load-store loop would wait out one memory latency per element)
    if (!a.tma_tables) {
      const uint16_t* SC = static_cast<const uint16_t*>(a.scales);
      const int ns = ng * (BN / 2);
      for (int i0 = tid; i0 < ns; i0 += 4 * nthr) {
        uint32_t v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = i0 + j * nthr, gr = i / (BN / 2), c = 2 * (i % (BN / 2));
          v[j] = (i < ns && n0 + c < N) ? *reinterpret_cast<const uint32_t*>(SC + size_t(g0 + gr) * N + n0 + c) : 0u;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (i0 + j * nthr < ns) reinterpret_cast<uint32_t*>(scl)[i0 + j * nthr] = v[j];
      }
      if (HAS_Z) {
        const int nz = ng * (BN / 8);
        for (int i0 = tid; i0 < nz; i0 += 4 * nthr) {
          uint32_t v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * nthr, gr = i / (BN / 8), c = i % (BN / 8);
            v[j] = (i < nz && n0 + 8 * c < N)
                       ? static_cast<uint32_t>(a.qzeros[size_t(g0 + gr) * (N / 8) + n0 / 8 + c]) : 0u;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (i0 + j * nthr < nz) zp[i0 + j * nthr] = v[j];
        }
      }
    }
    {
      if (!PERM)  // the zero row after each 256-value half of every x stage
        for (int i = tid; i < NS * 2 * 128; i += nthr) {
          const int st = i / 256, h = (i / 128) % 2, c = i % 128;
          reinterpret_cast<uint32_t*>(xst + size_t(st) * xstage)[(h * (MT + 1) + MT) * 128 + c] = 0u;
        }
    }
    if (PERM) {  // rows M .. MT-1, the zero row MT and the tail of the gathered x read as zero
      const int kr = kUnitK * (u1 - u0);
      for (int i = tid; i < (MT + 1) * krp; i += nthr) {
        const int m = i / krp, kk = i % krp;
        if (m >= M || kk >= kr) xg[i] = 0;
      }
    }
    pdl_wait();
    if (PERM && u1 > u0) {
      // x of this CTA's K-slice in sorted order: xg[m][i] = x[m, perm[64 u0 + i]],
      // gathered once; the indices are already in shared memory, so the loads
      // of a thread are independent and overlap
      if (!mbar_wait(pbar, 0)) *cfailed = 1;
      const uint16_t* X = static_cast<const uint16_t*>(a.x);
      const int32_t* pvs = reinterpret_cast<const int32_t*>(smem + L.pv);
      const int kr = kUnitK * (u1 - u0);
      for (int m = 0; m < M; ++m) {
        const uint16_t* Xm = X + size_t(m) * K;
        for (int i0 = tid; i0 < kr; i0 += 4 * nthr) {
          uint16_t v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * nthr;
            v[j] = i < kr ? Xm[min(max(pvs[i], 0), K - 1)] : 0;  // clamped: never read out of bounds
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // stored in the MMA's pair order: within each 8 values of k, (x0, x4),
            // (x1, x5), (x2, x6), (x3, x7) -- one 16-byte load per word row then
            // gives the four B registers without any byte permutes
            const int i = i0 + j * nthr;
            if (i < kr) xg[size_t(m) * krp + (i & ~7) + 2 * (i & 3) + ((i >> 2) & 1)] = v[j];
          }
        }
      }
    }
    consumer_sync(nthr);  // tables (and the gathered x) complete before any warp uses them
    if (a.tma_tables && u1 > u0 && !mbar_wait(tbar, 0)) *cfailed = 1;

    const int g = lane >> 2, t = lane & 3;
    const int slab = warp / KW, kpart = warp % KW;
    const int col4 = slab * kSlabCols + 4 * g;  // this thread's 4 columns within the tile
    const bool slab_live = !TILED || slab < nvalid;
    // x row of this lane's B fragment in n-tile nt (MT: the zero row; with
    // several n-tiles MT = 8 NT and rows past M are TMA zero fill)
    const int xrow = g < MT ? g : MT;
    const int ub = kpart * UPW;  // first unit of this warp within a stage

    // acc: running sums (scale applied); tmp: the current group's MMA sums
    float acc[2][NT][4], tmp[2][NT][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[j][nt][i] = tmp[j][nt][i] = 0.f;
    int cur_g = -1;
    // per column of the thread: pair of -(1024 + z) (fp16) or -(128 + z) (bf16),
    // and (fp16) pair of -(64 + z); z = 8 without stored zeros
    uint32_t zsv[4], zfv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      zsv[c] = ACT_BF16 ? 0xC308C308u : 0xE408E408u;
      zfv[c] = 0xD480D480u;
    }

    auto fold = [&](int gi) {  // acc += s(group) * tmp; tmp = 0
      const uint2 sb = *reinterpret_cast<const uint2*>(scl + gi * BN + col4);
      const float sv[4] = {ACT_BF16 ? bf16_bits_to_f32(sb.x & 0xFFFFu) : f16_bits_to_f32(sb.x & 0xFFFFu),
                           ACT_BF16 ? bf16_bits_to_f32(sb.x >> 16) : f16_bits_to_f32(sb.x >> 16),
                           ACT_BF16 ? bf16_bits_to_f32(sb.y & 0xFFFFu) : f16_bits_to_f32(sb.y & 0xFFFFu),
                           ACT_BF16 ? bf16_bits_to_f32(sb.y >> 16) : f16_bits_to_f32(sb.y >> 16)};
#pragma unroll
      for (int tl = 0; tl < 2; ++tl)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[tl][nt][i] = fmaf(sv[2 * tl + (i >> 1)], tmp[tl][nt][i], acc[tl][nt][i]);
            tmp[tl][nt][i] = 0.f;
          }
    };

    int s = 0;
    uint32_t ph = 0;  // parity of the full phase awaited in slot s
    for (int it = 0; it < n_stages; ++it) {
      if (!mbar_wait_sleep(&full[s], ph)) *cfailed = 1;
      if (*cfailed) break;
      const int nu = min(kStageUnits, u1 - u0 - kStageUnits * it);
      const uint8_t* xs = xst + size_t(s) * xstage;
      const uint8_t* wst = ring + size_t(s) * stage_w;
      if (slab_live) {
#pragma unroll
        for (int uu = 0; uu < UPW; ++uu) {
          const int ul = ub + uu;  // unit within the stage
          if (ul >= nu) break;
          const int u = u0 + kStageUnits * it + ul;
          const int gi = (u >> a.gshift) - g0;
          if (gi != cur_g) {  // a new scale group: apply the finished one, set up the new zeros
            if (cur_g >= 0) fold(cur_g);
            cur_g = gi;
            if (HAS_Z) {
              // fp16 -(1024 + z) = 0xE400 + z, -(64 + z) = 0xD400 + 16 z; bf16 -(128 + z) = 0xC300 + z,
              // both halves at once: z * 0x00010001 + the pair of the constant
              const uint32_t zw = zp[gi * (BN / 8) + col4 / 8] >> (4 * (col4 % 8));
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const uint32_t z = (zw >> (4 * c)) & 15u;
                zsv[c] = z * 0x00010001u + (ACT_BF16 ? 0xC300C300u : 0xE400E400u);
                zfv[c] = z * 0x00100010u + 0xD400D400u;
              }
            }
          }
          // the unit's 1 KB block of this slab: [unit][slab] (tiled) or [slab][unit] (GPTQ boxes)
          const uint8_t* ublk = TILED ? wst + (size_t(ul) * nslab + slab) * kUnitBytes
                                      : wst + size_t(slab) * kSlabStageBytes + ul * kUnitBytes;
          // x of the unit: the stage's half ul / 4 (x staged per stage) or the gathered slice
          const uint8_t* xu = PERM ? reinterpret_cast<const uint8_t*>(
                                         xg + size_t(xrow) * krp + kUnitK * (kStageUnits * it + ul))
                                   : xs + (((ul >> 2) * (MT + 1) + xrow) * 256 + kUnitK * (ul & 3)) * 2;
#pragma unroll
          for (int ab = 0; ab < 2; ++ab) {
            const int rr = 2 * t + ab;  // word row within the unit
            const uint4 wv = TILED ? *reinterpret_cast<const uint4*>(ublk + ab * 512 + lane * 16)
                                   : *reinterpret_cast<const uint4*>(ublk + rr * 128 + (((g ^ rr) & 7) << 4));
            // B registers of each n-tile: the x pairs (x0, x4), (x1, x5), (x2, x6),
            // (x3, x7) of the word row (the gathered act-order x is stored in that
            // order already); n-tile nt reads row 8 nt + g, 16 * 256 bytes further on
            uint32_t bx[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint4 xv = *reinterpret_cast<const uint4*>(xu + rr * 16 + nt * (8 * 256 * 2));
              bx[nt][0] = PERM ? xv.x : prmt(xv.x, xv.z, 0x5410u);
              bx[nt][1] = PERM ? xv.y : prmt(xv.x, xv.z, 0x7632u);
              bx[nt][2] = PERM ? xv.z : prmt(xv.y, xv.w, 0x5410u);
              bx[nt][3] = PERM ? xv.w : prmt(xv.y, xv.w, 0x7632u);
            }
            const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int tl = 0; tl < 2; ++tl) {
              const uint32_t we = w4[2 * tl], wo = w4[2 * tl + 1];
              const uint32_t we8 = we >> 8, wo8 = wo >> 8;
              const uint32_t zse = zsv[2 * tl], zso = zsv[2 * tl + 1], zfe = zfv[2 * tl], zfo = zfv[2 * tl + 1];
              const uint32_t q0 = convert_pair<ACT_BF16, 0>(we, we8, zse, zfe), q1 = convert_pair<ACT_BF16, 0>(wo, wo8, zso, zfo);
              const uint32_t q2 = convert_pair<ACT_BF16, 1>(we, we8, zse, zfe), q3 = convert_pair<ACT_BF16, 1>(wo, wo8, zso, zfo);
              const uint32_t q4 = convert_pair<ACT_BF16, 2>(we, we8, zse, zfe), q5 = convert_pair<ACT_BF16, 2>(wo, wo8, zso, zfo);
              const uint32_t q6 = convert_pair<ACT_BF16, 3>(we, we8, zse, zfe), q7 = convert_pair<ACT_BF16, 3>(wo, wo8, zso, zfo);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                mma_16816<ACT_BF16>(tmp[tl][nt], q0, q1, q2, q3, bx[nt][0], bx[nt][1]);
                mma_16816<ACT_BF16>(tmp[tl][nt], q4, q5, q6, q7, bx[nt][2], bx[nt][3]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == NS) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (cur_g >= 0) fold(cur_g);

    // ------------------------------------------------ split-K partial sums out
    // this thread holds rows m = 8 nt + 2t, 8 nt + 2t + 1 of columns col4 ..
    // col4 + 3; the owner of slab w is cluster rank w % S, slot (sender, kpart, w / S, m)
    const int owner = slab % S, lslab = slab / S;
    auto slot = [&](int sender, int m) {
      return recv + ((size_t(sender * KW + kpart) * nown_max + lslab) * MT + m) * kSlabCols + 4 * g;
    };
    if (S == 1) {
      consumer_sync(nthr);  // the pieces overwrite the ring: every consumer is past its last stage
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const int m = 8 * nt + 2 * t + p;
          if (m < MT)
            *reinterpret_cast<float4*>(slot(0, m)) =
                make_float4(acc[0][nt][p], acc[0][nt][2 + p], acc[1][nt][p], acc[1][nt][2 + p]);
        }
      mbar_arrive(recv_bar);  // release: the stores above are visible to the waiter
    } else {
      __syncwarp();
      cluster_wait();
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const int m = 8 * nt + 2 * t + p;
          if (m < MT)
            st_async_v4_to_rank(smem_u32(slot(int(rank), m)), acc[0][nt][p], acc[0][nt][2 + p], acc[1][nt][p],
                                acc[1][nt][2 + p], smem_u32(recv_bar), uint32_t(owner));
        }
    }
  }

  // ---------------------------------------------- owner: sum the pieces, store y
  if (nown > 0 && mbar_wait(recv_bar, 0)) {
    uint16_t* Y = static_cast<uint16_t*>(a.y);
    const int per = M * kSlabCols;
    for (int e = threadIdx.x; e < nown * per; e += blockDim.x) {
      const int i = e / per, m = (e % per) / kSlabCols, c = e % kSlabCols;
      const int n = n0 + (int(rank) + S * i) * kSlabCols + c;
      float v = 0.f;
      for (int sender = 0; sender < S; ++sender)
        for (int j = 0; j < KW; ++j)
          v += recv[((size_t(sender * KW + j) * nown_max + i) * MT + m) * kSlabCols + c];
      if (n < N) Y[size_t(m) * N + n] = f32_to_act<ACT_BF16>(v);
    }
  }
}

struct Problem4T {
  const void* x;
  const int32_t* qweight;
  const uint8_t* wtiled;
  const void* scales;
  const int32_t* qzeros;
  const int32_t* perm;
  void* y;
  int M, K, N, group, gshift;
  unsigned flags;
  cudaStream_t stream;
};

// Values of k of the largest of S K-slices (a multiple of 64).
int krange_max(int units, int S) { return kUnitK * ((units + S - 1) / S); }

int groups_per_slice_max(int units, int S, int group) {
  int ng_max = 1;
  for (int s = 0; s < S; ++s) {
    const int u0 = static_cast<int>((static_cast<long long>(s) * units) / S);
    const int u1 = static_cast<int>((static_cast<long long>(s + 1) * units) / S);
    if (u1 > u0) ng_max = std::max(ng_max, (kUnitK * u1 - 1) / group - (kUnitK * u0) / group + 1);
  }
  return ng_max;
}

// Plan and launch one kernel instance.  Candidate tiles (nslab slabs, S
// K-slices) are tried from the least work per CTA up; the first whose grid
// runs in one wave (all T clusters resident at once -- on GB300 the SMs sit in
// GPCs, so a cluster size that does not divide a GPC leaves SMs idle) is used.
template <int ACT, bool HZ, bool PERM, bool TILED, int NT>
cudaError_t launch_4t(const Problem4T& pr) {
  const void* kern = reinterpret_cast<const void*>(k4t_gemv_kernel<ACT, HZ, PERM, TILED, NT>);
  const int units = pr.K / kUnitK;
  const int MT = NT > 1 ? 8 * NT : pr.M <= 1 ? 1 : pr.M <= 2 ? 2 : pr.M <= 4 ? 4 : 8;
  const int max_slabs = PERM ? kMaxSlabsPerm : (NT == 4 ? 6 : 8);  // the kernel's thread bound
  const int max_smem = device_max_smem();
  struct Cand { long long cost; int S, nslab; };
  Cand cands[5 * 8];
  int nc = 0;
  for (int nslab = 4; nslab <= max_slabs; ++nslab)
    for (int S = 1; S <= 8 && S <= units; ++S)
      cands[nc++] = Cand{static_cast<long long>(nslab) * ((units + S - 1) / S), S, nslab};
  std::sort(cands, cands + nc, [](const Cand& a, const Cand& b) {
    return a.cost != b.cost ? a.cost < b.cost : (a.S != b.S ? a.S < b.S : a.nslab > b.nslab);
  });
  Plan4T q{0, 0, 0, 0, MT};
  size_t smem = 0;
  int ng_max = 1;
  for (int i = 0; i < nc && q.nslab == 0; ++i) {
    const int nslab = cands[i].nslab, S = cands[i].S;
    const int T = (pr.N + nslab * kSlabCols - 1) / (nslab * kSlabCols);
    if (T * S > device_sm_count()) continue;
    const int ng = groups_per_slice_max(units, S, pr.group);
    const int kr = krange_max(units, S);
    // a three-stage ring; its shared memory (over half an SM's) also keeps two
    // CTAs of one launch off the same SM, while the CTA of a smaller kernel
    // launched next can still start beside it
    int NS = 3;
    size_t sm = Smem4T(nslab, NS, MT, S, ng, PERM, kr).total;
    while (sm > static_cast<size_t>(max_smem) && NS > 2) sm = Smem4T(nslab, --NS, MT, S, ng, PERM, kr).total;
    if (sm > static_cast<size_t>(max_smem)) continue;
    const int threads = (nslab * kw_of(PERM) + 1) * 32;
    // capacity counted at one CTA per SM (planning smem above half an SM's)
    if (T > cluster_capacity(kern, S, threads, std::max(sm, static_cast<size_t>(max_smem) / 2 + 1024))) continue;
    q = Plan4T{nslab, S, T, NS, MT};
    smem = sm;
    ng_max = ng;
  }
  if (q.nslab == 0) {  // more column tiles than fit at once: one K-slice, widest tile, several waves
    const int ng = groups_per_slice_max(units, 1, pr.group);
    int NS = 3;
    const int kr = krange_max(units, 1);
    size_t sm = Smem4T(max_slabs, NS, MT, 1, ng, PERM, kr).total;
    while (sm > static_cast<size_t>(max_smem) && NS > 2) sm = Smem4T(max_slabs, --NS, MT, 1, ng, PERM, kr).total;
    if (sm > static_cast<size_t>(max_smem)) return cudaErrorNotSupported;
    q = Plan4T{max_slabs, 1, (pr.N + max_slabs * kSlabCols - 1) / (max_slabs * kSlabCols), NS, MT};
    smem = sm;
    ng_max = ng;
  }
  const int threads = (q.nslab * kw_of(PERM) + 1) * 32;
  CUtensorMap wmap, wmap8, xmap;
  memset(&wmap, 0, sizeof wmap);
  memset(&wmap8, 0, sizeof wmap8);
  if (!TILED) {
    if (!encode_tensor_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, pr.qweight, pr.N, pr.K / 8, size_t(pr.N) * 4,
                              kSlabCols, kStageK / 8, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&wmap8, CU_TENSOR_MAP_DATA_TYPE_UINT32, pr.qweight, pr.N, pr.K / 8, size_t(pr.N) * 4,
                              kSlabCols, kUnitK / 8, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  memset(&xmap, 0, sizeof xmap);
  if (!PERM && !encode_tensor_map_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, pr.x, pr.K, pr.M, size_t(pr.K) * 2, 256,
                                     MT, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  // scale rows [K/group, N] (16-bit) and packed zero rows [K/group, N/8] (int32): one
  // box of ng_max rows each per CTA; the zeros' row pitch (N/2 bytes) must be a
  // multiple of 16 and the scale box at most 256 rows
  CUtensorMap smap, zmap;
  memset(&smap, 0, sizeof smap);
  memset(&zmap, 0, sizeof zmap);
  const int G = pr.K / pr.group;
  bool tma_tables = ng_max <= 256 && (!HZ || (pr.N / 2) % 16 == 0);
  if (tma_tables)
    tma_tables = encode_tensor_map_2d(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT16, pr.scales, pr.N, G, size_t(pr.N) * 2,
                                      q.nslab * kSlabCols, ng_max, CU_TENSOR_MAP_SWIZZLE_NONE) &&
                 (!HZ || encode_tensor_map_2d(&zmap, CU_TENSOR_MAP_DATA_TYPE_INT32, pr.qzeros, pr.N / 8, G,
                                              size_t(pr.N / 8) * 4, q.nslab * kSlabCols / 8, ng_max,
                                              CU_TENSOR_MAP_SWIZZLE_NONE));
  Args4T a{pr.x, pr.y, pr.scales, pr.qzeros, pr.wtiled, pr.perm, pr.M, pr.K, pr.N, pr.group, MT, q.nslab, q.NS,
           ng_max, pr.gshift, krange_max(units, q.S), tma_tables ? 1 : 0};
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(q.S, q.T, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = pr.stream;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (q.S > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = q.S;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pr.flags & WQ_FLAG_PDL) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  void* args[6] = {&wmap, &wmap8, &xmap, &smap, &zmap, &a};
  return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace

// ---------------------------------------------------------------------- host --

int wq4t_unit_k() { return kUnitK; }

cudaError_t launch_wq4t(const void* x, const int32_t* qweight, const uint8_t* wtiled, const void* scales,
                        const int32_t* qzeros, const int32_t* perm, void* y, int M, int K, int N, int group,
                        int act_bf16, unsigned flags, cudaStream_t stream) {
  int gshift = 0;
  while ((kUnitK << gshift) < group) ++gshift;
  const bool tiled = wtiled != nullptr, is_perm = perm != nullptr, hz = qzeros != nullptr;
  // M <= 8: one n-tile; 9 .. 32 rows (GPTQ layout, contiguous groups): two or four
  if ((kUnitK << gshift) != group || K % kUnitK != 0 || M < 1 || M > ((tiled || is_perm) ? 8 : 32))
    return cudaErrorNotSupported;
  const Problem4T pr{x, qweight, wtiled, scales, qzeros, perm, y, M, K, N, group, gshift, flags, stream};
#define WQ4T_LAUNCH(ACT, HZ, PERM, TILED) \
  if (act_bf16 == ACT && hz == HZ && is_perm == PERM && tiled == TILED) return launch_4t<ACT, HZ, PERM, TILED, 1>(pr);
#define WQ4T_LAUNCH_NT(ACT, HZ)                                                  \
  if (act_bf16 == ACT && hz == HZ && !is_perm && !tiled)                         \
    return M <= 16 ? launch_4t<ACT, HZ, false, false, 2>(pr) : launch_4t<ACT, HZ, false, false, 4>(pr);
  if (M > 8) {
    WQ4T_LAUNCH_NT(0, false) WQ4T_LAUNCH_NT(0, true) WQ4T_LAUNCH_NT(1, false) WQ4T_LAUNCH_NT(1, true)
    return cudaErrorInvalidValue;
  }
  WQ4T_LAUNCH(0, false, false, false) WQ4T_LAUNCH(0, false, false, true)
  WQ4T_LAUNCH(0, false, true, false) WQ4T_LAUNCH(0, false, true, true)
  WQ4T_LAUNCH(0, true, false, false) WQ4T_LAUNCH(0, true, false, true)
  WQ4T_LAUNCH(0, true, true, false) WQ4T_LAUNCH(0, true, true, true)
  WQ4T_LAUNCH(1, false, false, false) WQ4T_LAUNCH(1, false, false, true)
  WQ4T_LAUNCH(1, false, true, false) WQ4T_LAUNCH(1, false, true, true)
  WQ4T_LAUNCH(1, true, false, false) WQ4T_LAUNCH(1, true, false, true)
  WQ4T_LAUNCH(1, true, true, false) WQ4T_LAUNCH(1, true, true, true)
#undef WQ4T_LAUNCH_NT
#undef WQ4T_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace wq
