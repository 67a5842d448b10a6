// wq_gemv3t.cu -- 3-bit skinny GEMM (wq3_gemv at 3 <= M <= 8) with
// per-column fp16 scale and stored zero, on the warp-level tensor-core MMA
// (mma.sync m16n8k16, fp16 operands, fp32 accumulate).  One MMA serves all M
// rows, so the work per code does not grow with M as it does on CUDA cores
// (chained 4096 x 4096: 9.4 against 14.8 us at M = 4, 15.1 against 21.7 us at
// M = 8; at M <= 2 the CUDA-core kernel of wq_gemv3.cu is faster).
//
// Definition (GPTQ CUDA kernel walkthrough, CUDA核函數設計與實現):
//   y[m,n] = sum_k x[m,k] * (s[n] * q(k,n) - zero[n]),  zero[n] = s[n] * z[n] stored,
// evaluated as  y = s[n] * (sum_k x q) - zero[n] * (sum_k x).
// Storage: int32 [3K/32, N]; the 32 codes of k = 32b .. 32b+31 of a column
// form a 96-bit little-endian stream over word rows 3b .. 3b+2, code j at
// bits [3j, 3j+3).
//
// Code pairs.  One LOP3, (V & mask) | 0x6400_6400, turns a 32-bit window V of
// the stream into the fp16 pair (1024 + q_a 2^oa, 1024 + q_b 2^ob) whenever V
// holds code a at bit oa <= 7 and code b at bit 16 + ob, ob <= 7 (the codes
// land inside the 10-bit mantissas).  One HFMA2 by (2^-oa, 2^-ob) plus
// (-1024 2^-oa, -1024 2^-ob) then leaves (q_a, q_b) exactly.  The 32 codes of
// a block split into 16 such pairs over seven windows: the three words and
// four shifted ones, starting at stream bits 6, 12, 41 and 71 (found by an
// exhaustive search over pairings, which also shows that three shifted
// windows cannot cover a block).  Per code that is 5/8 of a logic op and 1/2
// of a packed-half op (the two pipes issue side by side); extracting each
// code to bit 0 costs about 1.3 logic ops.
//
// Fragments.  A = codes (16 columns x 16 k), B = x^T (16 k x 8 rows m).  The
// order of k inside one MMA is free, so the k slots of thread (g = lane/4,
// t = lane%4) hold two code pairs of one block: per unit of four blocks,
// thread t takes block t for columns 4g .. 4g+3 of the warp's 32-column slab
// (tile 0: columns 4g, 4g+1 as MMA rows g, g+8; tile 1: 4g+2, 4g+3), and its
// B registers are the x values of the same pairs.  The CTA lays its K-slice
// of x out in that pair order once, right after the dependency wait, and adds
// up x per unit on the way (the zero term).
//
// Weights go straight from HBM into the registers that convert them: per
// unit a thread loads its block's three word rows of its four columns, three
// 16-byte loads, and the eight lanes of one row read 128 contiguous bytes.
// Each code is used by one MMA only, so staging the weights in shared memory
// buys no reuse; a warp's share here is small (two units at 4096 x 4096), so
// all of its loads are in flight before the dependency wait (weights do not
// depend on the previous kernel), later ones two units ahead.
//
// A CTA is small -- 8 warps, at most 112 registers a thread, a few KB of
// shared memory -- so that it fits on an SM beside the CTAs of the kernel
// launched before it: with programmatic dependent launch it then starts, and
// has its weights in registers, while that kernel is still running.  After
// the wait, x of the CTA's K-slice arrives by one bulk copy per row (through
// the TMA engine: per-thread loads of x queued behind the weight loads took
// ~1 us), and each warp lays out the x of its own units in pair order
// (shared memory rows an odd multiple of 64 bytes apart, 16-byte chunk q of
// block b at q ^ (b % 4): the B loads are conflict-free), adding up x per unit
// on the way (the zero term); no CTA-wide barrier follows.
//
// Work decomposition: a CTA owns nslab 32-column slabs and a K-slice of
// 128-value units; each warp a contiguous run of units of one slab; the S CTAs
// of a cluster add their partial sums through distributed shared memory.
#include <algorithm>
#include <cstring>

#include "../../include/wq.h"
#include "wq_gemv_common.cuh"
#include "wq_launch.h"

namespace wq {

namespace {

constexpr int kSlabCols = 32;
constexpr int kBlockK = 32;                    // codes of one 3-word block
constexpr int kUnitK = 4 * kBlockK;            // a unit: one block per thread t
constexpr int kWarps3 = 8;
constexpr int kThreads3 = kWarps3 * 32;
constexpr int kMaxRegs3 = 112;  // two CTAs of 288 threads x 64 registers leave room for one of these

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

// ------------------------------------------------------------ the pair cover
// Pair p (0 .. 15) holds codes (pair_a(p), pair_b(p)) of a block, read from
// the window that starts at stream bit pair_window(p).
__host__ __device__ constexpr int pair_a(int p) { return p < 6 ? p : (p < 11 ? p + 6 : p + 11); }
__host__ __device__ constexpr int pair_b(int p) { return pair_a(p) + (p < 6 ? 6 : 5); }
__host__ __device__ constexpr int pair_window(int p) {
  return p < 2 ? 0 : p < 4 ? 6 : p < 6 ? 12 : p < 8 ? 32 : p < 11 ? 41 : p < 13 ? 64 : 71;
}
__host__ __device__ constexpr int window_slot(int s) {
  return s == 0 ? 0 : s == 6 ? 1 : s == 12 ? 2 : s == 32 ? 3 : s == 41 ? 4 : s == 64 ? 5 : 6;
}
__host__ __device__ constexpr int pair_oa(int p) { return 3 * pair_a(p) - pair_window(p); }
__host__ __device__ constexpr int pair_ob(int p) { return 3 * pair_b(p) - pair_window(p) - 16; }
// position of code j in the pair-ordered x of its block: 2 p + (j is the pair's second code)
__host__ __device__ constexpr int pair_pos(int j) {
  int r = 0;
  for (int p = 0; p < 16; ++p) {
    if (pair_a(p) == j) r = 2 * p;
    if (pair_b(p) == j) r = 2 * p + 1;
  }
  return r;
}
// the eight positions of codes 8q .. 8q+7, 5 bits each
__host__ __device__ constexpr uint64_t pair_pos_row(int q) {
  uint64_t v = 0;
  for (int e = 0; e < 8; ++e) v |= uint64_t(pair_pos(8 * q + e)) << (5 * e);
  return v;
}
constexpr uint64_t kPosRow0 = pair_pos_row(0), kPosRow1 = pair_pos_row(1), kPosRow2 = pair_pos_row(2),
                   kPosRow3 = pair_pos_row(3);
constexpr bool pair_cover_ok() {
  uint32_t seen = 0;
  for (int p = 0; p < 16; ++p) {
    const int oa = pair_oa(p), ob = pair_ob(p);
    if (oa < 0 || oa > 7 || ob < 0 || ob > 7) return false;
    seen |= (1u << pair_a(p)) | (1u << pair_b(p));
  }
  return seen == 0xFFFFFFFFu;
}
static_assert(pair_cover_ok(), "16 pairs, every code once, each inside the fp16 mantissas of its window");

// fp16 bits of 2^-o and of -1024 * 2^-o
__host__ __device__ constexpr uint32_t h_pow2m(int o) { return uint32_t(15 - o) << 10; }
__host__ __device__ constexpr uint32_t h_negbias(int o) { return 0x8000u | (uint32_t(25 - o) << 10); }

__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<const __half2*>(&u); }
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }

// The seven windows of one column's block (w0, w1, w2 = its three words).
__device__ __forceinline__ void block_windows(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t (&v)[7]) {
  v[0] = w0;
  v[1] = w0 >> 6;
  v[2] = shf_r(w0, w1, 12);
  v[3] = w1;
  v[4] = shf_r(w1, w2, 9);
  v[5] = w2;
  v[6] = w2 >> 7;
}

// Codes of pair p as the exact fp16 pair (q_a, q_b).  p is a constant after unrolling.
__device__ __forceinline__ uint32_t code_pair(const uint32_t (&v)[7], int p) {
  const int oa = pair_oa(p), ob = pair_ob(p);
  const uint32_t m = lop3_and_or(v[window_slot(pair_window(p))], (7u << oa) | (7u << (16 + ob)), 0x64006400u);
  return h2_bits(__hfma2(as_h2(m), as_h2(h_pow2m(oa) | (h_pow2m(ob) << 16)),
                         as_h2(h_negbias(oa) | (h_negbias(ob) << 16))));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16 bytes of packed weights, read once: not kept in L1.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Bytes global -> this CTA's shared memory by the TMA engine, completing on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

struct Args3T {
  const void* x;
  const int32_t* mat;
  void* y;
  const void* scales;
  const void* zeros;
  int M, K, N;
  int nslab;
  int kur;  // units of the largest K-slice
};

struct Smem3T {
  size_t xraw, xg, xsu, recv, bar, total;
  // row pitch of the pair-ordered x, in values: an odd multiple of 32 (64 bytes)
  __host__ __device__ static int xpitch(int kur) { return kur * kUnitK + 32; }
  __host__ __device__ Smem3T(int nslab, int M, int S, int kur) {
    const int KW = kWarps3 / nslab, nown = (nslab + S - 1) / S;
    size_t o = 0;
    xraw = o;  o = align16(o + size_t(M) * kur * kUnitK * 2);  // x slice as stored (one bulk copy per row)
    xg = o;    o = align16(o + size_t(M) * xpitch(kur) * 2);
    xsu = o;   o = align16(o + size_t(M) * kur * 4);
    recv = o;  o = align16(o + size_t(S) * KW * nown * M * kSlabCols * 4);
    bar = o;   o = align16(o + 16);  // recv_bar, xbar
    total = o;
  }
};

// One unit's weights of this thread: word rows 3b .. 3b+2 of block b = 4u + t,
// columns col4 .. col4+3 (zeros past K or N).
struct UnitWords {
  uint32_t w[3][4];
};
__device__ __forceinline__ void load_unit(UnitWords& r, const int32_t* mat, int N, int nblk, int u, int t, int col4) {
  const int b = 4 * u + t;
  const bool live = b < nblk && col4 < N;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    uint4 q = make_uint4(0u, 0u, 0u, 0u);
    if (live) q = ldg_stream(mat + (size_t(3 * b + i) * N + col4));
    r.w[i][0] = q.x;
    r.w[i][1] = q.y;
    r.w[i][2] = q.z;
    r.w[i][3] = q.w;
  }
}

__global__ void __maxnreg__(kMaxRegs3) k3t_gemv_kernel(const Args3T a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int S = gridDim.x;
  const int nslab = a.nslab, M = a.M, K = a.K, N = a.N;
  const int KW = kWarps3 / nslab;  // warps per slab (a power of two)
  const Smem3T L(nslab, M, S, a.kur);
  uint16_t* xg = reinterpret_cast<uint16_t*>(smem + L.xg);
  float* xsu = reinterpret_cast<float*>(smem + L.xsu);
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  uint64_t* recv_bar = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* xbar = recv_bar + 1;  // the x slice
  const uint16_t* xraw = reinterpret_cast<const uint16_t*>(smem + L.xraw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int n0 = blockIdx.y * nslab * kSlabCols;
  const int nblk = K / kBlockK;
  const int units = (nblk + 3) / 4;
  int u0, u1;
  split_range(units, S, blockIdx.x, u0, u1);
  const uint32_t rank = S > 1 ? cluster_rank() : 0u;
  const int nown_max = (nslab + S - 1) / S;
  const int nown = int(rank) < nslab ? (nslab - int(rank) + S - 1) / S : 0;
  const int xp = Smem3T::xpitch(a.kur);
  const int slab = warp / KW, kpart = warp % KW;
  const int col4 = n0 + slab * kSlabCols + 4 * g;  // this thread's 4 columns (N % 8 == 0: all or none exist)
  // this warp's units: a contiguous run [ua, ub) of the slice
  const int nu = u1 - u0, per = (nu + KW - 1) / KW;
  const int ua = u0 + min(nu, kpart * per), ub = u0 + min(nu, (kpart + 1) * per);
  const int nmine = ub - ua;

  if (threadIdx.x == 0) {
    mbar_init(xbar, 1);
    if (S == 1) {
      mbar_init(recv_bar, kThreads3);
    } else {
      mbar_init(recv_bar, 1);
      const uint32_t rb = uint32_t(S) * KW * nown * M * kSlabCols * 4;
      if (rb) mbar_expect_tx(recv_bar, rb);
    }
    fence_mbar_init();
  }
  // weights, scale and stored zero are not written by the previous kernel:
  // read them before the dependency wait
  UnitWords wr[2];
  if (nmine > 0) load_unit(wr[0], a.mat, N, nblk, ua, t, col4);
  if (nmine > 1) load_unit(wr[1], a.mat, N, nblk, ua + 1, t, col4);
  // (raw bits: nothing waits for these loads before the epilogue)
  uint2 sv = make_uint2(0u, 0u), zv = make_uint2(0u, 0u);
  if (col4 < N) {
    sv = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.scales) + col4);
    zv = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.zeros) + col4);
  }
  __syncthreads();  // recv_bar initialised
  if (S > 1) cluster_arrive_relaxed();
  pdl_launch_dependents();
  pdl_wait();
  // x of the CTA's K-slice as stored: one bulk copy per row (the TMA engine,
  // not the warps' load queues, which still hold the weight loads issued
  // before the wait: loads of x queued behind them took ~1 us)
  const int k0 = u0 * kUnitK;
  const int kcopy = max(0, min(nu * kUnitK, K - k0));  // values of the slice that exist (a multiple of 32)
  if (threadIdx.x == 0 && kcopy > 0) {
    mbar_expect_tx(xbar, uint32_t(M) * kcopy * 2);
    for (int m = 0; m < M; ++m)
      bulk_copy_g2s(smem + L.xraw + size_t(m) * a.kur * kUnitK * 2, static_cast<const uint16_t*>(a.x) + size_t(m) * K + k0,
                    uint32_t(kcopy) * 2, xbar);
  }
  const bool x_ok = kcopy == 0 || __all_sync(0xffffffffu, mbar_wait(xbar, 0));
  {
    // x of this warp's units in pair order, xg[m][b * 32 + pos] (b: block within
    // the slice) with 16-byte chunk q of block b at q ^ (b % 4), and the sum of x
    // per unit.  Lane l takes 8 values (chunk c): block c / 4, codes 8 (l % 4) ..
    // +7; the 32 lanes cover two units.  Only this warp reads what it writes.
    const int q4 = lane & 3;
    const uint64_t prow = q4 == 0 ? kPosRow0 : q4 == 1 ? kPosRow1 : q4 == 2 ? kPosRow2 : kPosRow3;
    const int c_lo = (ua - u0) * (kUnitK / 8), c_hi = (ub - u0) * (kUnitK / 8);
    for (int m = 0; m < M; ++m) {
      for (int c0 = c_lo; c0 < c_hi; c0 += 32) {  // warp-uniform trip count
        const int c = c0 + lane;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (x_ok && c < c_hi && 8 * c < kcopy)
          v = *reinterpret_cast<const uint4*>(xraw + size_t(m) * a.kur * kUnitK + 8 * c);
        const int b = c >> 2;
        uint16_t* dst = xg + size_t(m) * xp + size_t(b) * kBlockK;
        const uint32_t h[4] = {v.x, v.y, v.z, v.w};
        float sum = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint16_t xv = static_cast<uint16_t>(h[e >> 1] >> (16 * (e & 1)));
          const int pos = static_cast<int>((prow >> (5 * e)) & 31u);
          if (c < c_hi) dst[(((pos >> 3) ^ (b & 3)) << 3) | (pos & 7)] = xv;
          sum += f16_bits_to_f32(xv);
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if ((lane & 15) == 0 && c < c_hi) xsu[m * a.kur + (c >> 4)] = sum;
      }
    }
  }
  __syncwarp();

  float acc[2][2][4];
#pragma unroll
  for (int tl = 0; tl < 2; ++tl)
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[tl][h][i] = 0.f;
  float xw[2] = {0.f, 0.f};  // sum of x over this warp's units, rows 2t and 2t + 1
  const bool brow = g < M;   // lanes whose B column is a row of x (the others feed zeros)
  const uint8_t* xrow = reinterpret_cast<const uint8_t*>(xg + size_t(brow ? g : 0) * xp);

  auto unit_mma = [&](const UnitWords& r, int ul) {  // ul: unit within the slice
    const int bl = 4 * ul + t;                       // this thread's block within the slice
    uint32_t xb[16];
    {
      const uint8_t* xr = xrow + size_t(bl) * kBlockK * 2;
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        uint4 q = make_uint4(0u, 0u, 0u, 0u);
        if (brow) q = *reinterpret_cast<const uint4*>(xr + ((qq ^ (bl & 3)) << 4));
        xb[4 * qq] = q.x;
        xb[4 * qq + 1] = q.y;
        xb[4 * qq + 2] = q.z;
        xb[4 * qq + 3] = q.w;
      }
    }
#pragma unroll
    for (int p = 0; p < 2; ++p)
      if (2 * t + p < M) xw[p] += xsu[(2 * t + p) * a.kur + ul];
#pragma unroll
    for (int tl = 0; tl < 2; ++tl) {
      uint32_t ve[7], vo[7];  // windows of column 4g + 2tl (MMA row g) and 4g + 2tl + 1 (row g + 8)
      block_windows(r.w[0][2 * tl], r.w[1][2 * tl], r.w[2][2 * tl], ve);
      block_windows(r.w[0][2 * tl + 1], r.w[1][2 * tl + 1], r.w[2][2 * tl + 1], vo);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        mma_f16(acc[tl][i & 1], code_pair(ve, 2 * i), code_pair(vo, 2 * i), code_pair(ve, 2 * i + 1),
                code_pair(vo, 2 * i + 1), xb[2 * i], xb[2 * i + 1]);
    }
  };
  // two units in registers: compute one, then load the unit two ahead into its place
  for (int i = 0; i < nmine; i += 2) {
    unit_mma(wr[0], ua - u0 + i);
    if (i + 2 < nmine) load_unit(wr[0], a.mat, N, nblk, ua + i + 2, t, col4);
    if (i + 1 < nmine) {
      unit_mma(wr[1], ua - u0 + i + 1);
      if (i + 3 < nmine) load_unit(wr[1], a.mat, N, nblk, ua + i + 3, t, col4);
    }
  }

  // this warp's share of y: s (sum x q) - zero (sum x) over the k it handled;
  // thread holds rows m = 2t, 2t+1 of columns col4 .. col4 + 3
  const float sc[4] = {f16_bits_to_f32(sv.x & 0xFFFFu), f16_bits_to_f32(sv.x >> 16), f16_bits_to_f32(sv.y & 0xFFFFu),
                       f16_bits_to_f32(sv.y >> 16)};
  const float zr[4] = {f16_bits_to_f32(zv.x & 0xFFFFu), f16_bits_to_f32(zv.x >> 16), f16_bits_to_f32(zv.y & 0xFFFFu),
                       f16_bits_to_f32(zv.y >> 16)};
  float part[2][4];
#pragma unroll
  for (int tl = 0; tl < 2; ++tl)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = 2 * tl + (i >> 1);
      part[tl][i] = fmaf(sc[c], acc[tl][0][i] + acc[tl][1][i], -zr[c] * xw[i & 1]);
    }
  // the owner of slab w is cluster rank w % S, slot (sender, kpart, w / S, m)
  const int owner = slab % S, lslab = slab / S;
  auto slot = [&](int sender, int m) {
    return recv + ((size_t(sender * KW + kpart) * nown_max + lslab) * M + m) * kSlabCols + 4 * g;
  };
  if (S == 1) {
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int m = 2 * t + p;
      if (m < M)
        *reinterpret_cast<float4*>(slot(0, m)) = make_float4(part[0][p], part[0][2 + p], part[1][p], part[1][2 + p]);
    }
    mbar_arrive(recv_bar);  // release: the stores above are visible to the waiter
  } else {
    __syncwarp();
    cluster_wait();
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int m = 2 * t + p;
      if (m < M)
        st_async_v4_to_rank(smem_u32(slot(int(rank), m)), part[0][p], part[0][2 + p], part[1][p], part[1][2 + p],
                            smem_u32(recv_bar), uint32_t(owner));
    }
  }

  // ---------------------------------------------- owner: sum the pieces, store y
  // the S * KW pieces of an element are added by `lanes` neighbouring lanes
  // (a power of two up to 16), then in a fixed butterfly order
  // (every lane of a warp takes the same branch: the butterfly needs the whole warp)
  if (__all_sync(0xffffffffu, nown > 0 && mbar_wait(recv_bar, 0))) {
    __half* Y = static_cast<__half*>(a.y);
    const int npieces = S * KW, per = M * kSlabCols;
    int lanes = 1;
    while (2 * lanes <= npieces && 2 * lanes <= 16) lanes *= 2;
    const int total = nown * per * lanes;
    for (int base = warp * 32; base < total; base += kThreads3) {  // warp-uniform trip count
      const int e0 = base + lane, e = e0 / lanes, j0 = e0 % lanes;
      const int i = e / per, m = (e % per) / kSlabCols, c = e % kSlabCols;
      float v = 0.f;
      if (e0 < total)
        for (int j = j0; j < npieces; j += lanes) {
          const int sender = j / KW, kp = j % KW;
          v += recv[((size_t(sender * KW + kp) * nown_max + i) * M + m) * kSlabCols + c];
        }
      for (int o = 1; o < lanes; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      const int n = n0 + (int(rank) + S * i) * kSlabCols + c;
      if (e0 < total && j0 == 0 && n < N) Y[size_t(m) * N + n] = __float2half_rn(v);
    }
  }
  if (!x_ok && threadIdx.x == 0) mbar_wait(xbar, 0);  // a copy still in flight lands before the CTA exits
}

}  // namespace

// ---------------------------------------------------------------------- host --

// Plan: column tiles of nslab slabs (nslab in 1, 2, 4, 8; 8 / nslab warps per
// slab) and S K-slices.  A candidate's cost is its work per CTA times the CTAs
// an SM runs one after another (its grid over the SM count); among the
// cheapest, the least work per CTA (every warp's units are then requested
// before the dependency wait), then the smallest cluster.  Grids must be resident at once; if none is, one K-slice of 8-slab
// tiles in waves.  cudaErrorNotSupported: a shape this kernel does not take
// (M > 8, K % 32, N % 8, or shared memory for the pair-ordered x).
cudaError_t launch_wq3t(const void* x, const int32_t* mat, const void* scales, const void* zeros, void* y, int M,
                        int K, int N, unsigned flags, cudaStream_t stream) {
  if (M < 1 || M > 8 || K < kBlockK || K % kBlockK != 0 || N < 8 || N % 8 != 0) return cudaErrorNotSupported;
  const void* kern = reinterpret_cast<const void*>(k3t_gemv_kernel);
  const int units = (K / kBlockK + 3) / 4;
  const int max_smem = device_max_smem();
  const int sms = std::max(1, device_sm_count());
  struct Cand { long long cost, work; int S, nslab; };
  Cand cands[4 * 8];
  int nc = 0;
  for (int nslab = 1; nslab <= 8; nslab *= 2)
    for (int S = 1; S <= 8 && S <= units; ++S) {
      const long long t = (N + nslab * kSlabCols - 1) / (nslab * kSlabCols);
      const long long work = static_cast<long long>(nslab) * ((units + S - 1) / S);
      cands[nc++] = Cand{work * ((t * S + sms - 1) / sms), work, S, nslab};
    }
  std::sort(cands, cands + nc, [](const Cand& a, const Cand& b) {
    return a.cost != b.cost ? a.cost < b.cost : (a.work != b.work ? a.work < b.work : a.S < b.S);
  });
  int nslab = 0, S = 0, T = 0;
  size_t smem = 0;
  for (int i = 0; i < nc && nslab == 0; ++i) {
    const int ns = cands[i].nslab, s = cands[i].S;
    const int t = (N + ns * kSlabCols - 1) / (ns * kSlabCols);
    const size_t sm = Smem3T(ns, M, s, (units + s - 1) / s).total;
    if (sm > static_cast<size_t>(max_smem)) continue;
    if (t > cluster_capacity(kern, s, kThreads3, sm)) continue;  // the grid runs in one wave
    nslab = ns, S = s, T = t, smem = sm;
  }
  if (nslab == 0) {  // more column tiles than fit at once
    nslab = 8, S = 1, T = (N + 8 * kSlabCols - 1) / (8 * kSlabCols);
    smem = Smem3T(nslab, M, S, units).total;
    if (smem > static_cast<size_t>(max_smem)) return cudaErrorNotSupported;
  }
  Args3T a{x, mat, y, scales, zeros, M, K, N, nslab, (units + S - 1) / S};
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, T, 1);
  cfg.blockDim = dim3(kThreads3, 1, 1);
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
  void* args[1] = {&a};
  return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace wq
