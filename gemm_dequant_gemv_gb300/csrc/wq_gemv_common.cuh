// wq_gemv_common.cuh -- the skeleton shared by the CUDA-core GEMV kernels.
//
// Work decomposition (the same for every packed format):
//   * the weight matrix is cut into column tiles of BN columns (grid.y) and
//     the K dimension of each tile into S slices (grid.x).  The S CTAs of a
//     tile form one thread-block cluster and add their partial results
//     through distributed shared memory, so no partial sum goes to HBM;
//   * warp 8 of each CTA is the producer: one lane streams, per stage, a box
//     of packed weight rows and the matching box of x (all M rows) into a ring
//     of NS shared-memory stages with 2D TMA loads, gated by full/empty
//     mbarriers.  Weights are requested before griddepcontrol.wait, x after;
//   * warps 0..7 are consumers: per stage each converts its own slice of the
//     stage's x, takes one "unit" (a fixed number of packed rows), unpacks
//     the codes in registers, converts them with exact bit tricks and
//     accumulates in fp32 with packed FFMA2.  Warps run independently; only
//     the stage mbarriers order them.
#pragma once

#include "wq_device.cuh"

namespace wq {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kGemvThreads = kConsumerThreads + 32;

struct GemvArgs {
  const void* x;
  void* y;
  const void* scales;
  const void* zeros;     // 3-bit: fp16 stored zeros; 4-bit: packed qzeros (or null)
  const int32_t* g_idx;  // 4-bit act-order only
  int M, K, N, group;
  int ng_max;            // largest number of scale groups one CTA touches
};

// Balanced split of `units` work units into S slices; slice `s` = [u0, u1).
__device__ __forceinline__ void split_range(int units, int S, int s, int& u0, int& u1) {
  u0 = static_cast<int>((static_cast<long long>(s) * units) / S);
  u1 = static_cast<int>((static_cast<long long>(s + 1) * units) / S);
}

// Group index of work unit u (units of `unit_k` values of k, groups of `group`
// values, group a multiple of unit_k): a shift when the number of units per
// group is a power of two (the usual 64, 128, 256), a division otherwise.
struct UnitGroups {
  int per, shift;  // units per group; log2(per) or -1
  __device__ UnitGroups(int group, int unit_k) : per(group / unit_k) {
    shift = (per & (per - 1)) == 0 ? __ffs(per) - 1 : -1;
  }
  __device__ __forceinline__ int of(int u) const { return shift >= 0 ? (u >> shift) : u / per; }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Producer loop.  Stage `it` holds packed weight rows [wrow0 + it*wrows, +wrows)
// of column tile wcol0 (box of the weight map) and x columns
// [xcol0 + it*xcols, +xcols) for all rows (box of the x map), both completing
// on full[it % NS].  The weight boxes of the first NS stages are requested
// before the programmatic-dependency wait; every x box after it.
template <int NS>
__device__ __forceinline__ int produce_stages(const CUtensorMap* wmap, const CUtensorMap* xmap, uint8_t* wst,
                                              uint32_t wbytes, uint8_t* xst, uint32_t xbytes, uint64_t* full,
                                              uint64_t* empty, int wcol0, int wrow0, int wrows, int xcol0,
                                              int xcols, int n_loads, volatile int* cta_failed) {
  prefetch_tensormap(wmap);
  prefetch_tensormap(xmap);
  const uint64_t pol = l2_evict_first_policy();
  const int pre = n_loads < NS ? n_loads : NS;
  for (int it = 0; it < pre; ++it) {
    mbar_expect_tx(&full[it], wbytes + xbytes);
    tma_load_2d(wst + size_t(it) * wbytes, wmap, &full[it], wcol0, wrow0 + it * wrows, pol);
  }
  pdl_wait();
  for (int it = 0; it < pre; ++it) tma_load_2d(xst + size_t(it) * xbytes, xmap, &full[it], xcol0 + it * xcols, 0, 0ull);
  int issued = pre;
  for (int it = NS; it < n_loads; ++it) {
    const int s = it % NS;
    if (*cta_failed || !mbar_wait(&empty[s], ((it / NS) - 1) & 1)) {
      *cta_failed = 1;
      break;
    }
    mbar_expect_tx(&full[s], wbytes + xbytes);
    tma_load_2d(wst + size_t(s) * wbytes, wmap, &full[s], wcol0, wrow0 + it * wrows, pol);
    tma_load_2d(xst + size_t(s) * xbytes, xmap, &full[s], xcol0 + it * xcols, 0, 0ull);
    ++issued;
  }
  return issued;
}

// After a failed wait: let the copies already issued land before the CTA's
// shared memory goes away (each wait is itself bounded).
template <int NS>
__device__ __forceinline__ void drain_stages(uint64_t* full, int issued) {
  for (int s = 0; s < NS && s < issued; ++s) {
    const int last = ((issued - 1 - s) / NS) * NS + s;  // last load issued into stage s
    mbar_wait(&full[s], (last / NS) & 1);
  }
}

// As drain_stages, for a ring whose depth is a run-time value.
__device__ __forceinline__ void drain_stages_rt(uint64_t* full, int NS, int issued) {
  for (int s = 0; s < NS && s < issued; ++s) {
    const int last = ((issued - 1 - s) / NS) * NS + s;
    mbar_wait(&full[s], (last / NS) & 1);
  }
}

// Cross-warp / cross-CTA reduction without CTA-wide barriers.
//
// The tile's BN columns are split into S column chunks of `chunk` columns
// (a multiple of 4), chunk r owned by cluster rank r.  When a consumer warp
// has finished its K-slice, each lane sends its 4 columns (one 16-byte
// asynchronous remote store per row m) into slot (sender rank, warp) of the
// owner's receive buffer; the stores are counted on the owner's `recv_bar`,
// which was primed at start for all S * 8 pieces.  Each CTA then waits on its
// own recv_bar and adds, for its own columns, the S * 8 pieces in a fixed
// (rank, warp) order -- the result does not depend on timing -- and stores y.
// A cluster barrier (arrive at start, wait before the first remote store)
// makes sure every CTA's recv_bar is initialized before anything reaches it.
// Without a cluster (S == 1) the pieces are plain shared-memory stores and
// recv_bar counts one arrival per consumer thread instead of bytes.
struct TileReduce {
  int S, chunk;  // columns per owner (multiple of 4)
  __host__ __device__ TileReduce(int S_, int BN) : S(S_), chunk(((BN + S_ - 1) / S_ + 3) & ~3) {}
  __host__ __device__ int piece(int MT) const { return MT * chunk; }  // floats per (sender warp, owner)
  __host__ __device__ size_t recv_floats(int MT) const { return size_t(S) * kConsumerWarps * piece(MT); }
  // bytes one owner receives: S CTAs x 8 warps, MT rows of its columns
  __host__ __device__ uint32_t recv_bytes(int MT, int BN, int owner) const {
    const int len = min(chunk, BN - owner * chunk);
    return len > 0 ? uint32_t(S) * kConsumerWarps * MT * len * 4u : 0u;
  }
  // One thread, before the CTA's first cluster barrier arrive.
  __device__ void init_bar(uint64_t* recv_bar, int MT, int BN) const {
    if (S == 1) {
      mbar_init(recv_bar, kConsumerThreads);
      return;
    }
    mbar_init(recv_bar, 1);
    const uint32_t rb = recv_bytes(MT, BN, cluster_rank());
    if (rb) mbar_expect_tx(recv_bar, rb);
  }
};

// Consumer warp: send this warp's partial sums (columns 4*lane .. 4*lane+3 of
// the tile, MT rows) to their owner.  Waits first for the cluster barrier the
// CTA arrived on after initialising recv_bar.
template <int MT, int BN>
__device__ __forceinline__ void push_partials(const TileReduce& R, const float2 (*acc)[2], float* recv,
                                              uint64_t* recv_bar, int warp, int lane) {
  static_assert(BN == 128, "one column quad per lane");
  const int col = 4 * lane, r = col / R.chunk, cc = col % R.chunk;
  if (R.S == 1) {
    float* slot = recv + size_t(warp) * R.piece(MT);
#pragma unroll
    for (int m = 0; m < MT; ++m)
      *reinterpret_cast<float4*>(slot + m * R.chunk + cc) =
          make_float4(acc[m][0].x, acc[m][0].y, acc[m][1].x, acc[m][1].y);
    mbar_arrive(recv_bar);  // release: the stores above are visible to the waiter
    return;
  }
  __syncwarp();
  cluster_wait();
  const uint32_t me = cluster_rank();
  float* slot = recv + (size_t(me) * kConsumerWarps + warp) * R.piece(MT);
#pragma unroll
  for (int m = 0; m < MT; ++m)
    st_async_v4_to_rank(smem_u32(slot + m * R.chunk + cc), acc[m][0].x, acc[m][0].y, acc[m][1].x, acc[m][1].y,
                        smem_u32(recv_bar), uint32_t(r));
}

// Every thread of the CTA: wait for this CTA's pieces and store its columns.
template <int MT, int BN, class StoreFn>
__device__ __forceinline__ void owner_reduce_store(const TileReduce& R, const float* recv, uint64_t* recv_bar,
                                                   StoreFn store) {
  const uint32_t me = R.S > 1 ? cluster_rank() : 0u;
  const int c0 = int(me) * R.chunk;
  const int len = min(R.chunk, BN - c0);
  if (len <= 0) return;
  if (!mbar_wait(recv_bar, 0)) return;
  const int n_pieces = R.S * kConsumerWarps;
  for (int e = threadIdx.x; e < MT * len; e += blockDim.x) {
    const int m = e / len, cc = e % len;
    float v = 0.f;
    for (int p = 0; p < n_pieces; ++p) v += recv[size_t(p) * R.piece(MT) + m * R.chunk + cc];
    store(m, c0 + cc, v);
  }
}

// CTA-level reduction used by the tensor-core kernel: `part` holds this CTA's
// MT x BN partial tile; the S CTAs of the cluster each add up an equal share
// of the tile through distributed shared memory and store it.
template <int MT, int BN, class StoreFn>
__device__ __forceinline__ void finish_tile(const float* part, int S, StoreFn store) {
  constexpr int total = MT * BN;
  if (S == 1) {
    __syncthreads();
    for (int e = threadIdx.x; e < total; e += blockDim.x) store(e / BN, e % BN, part[e]);
    return;
  }
  cluster_sync();
  const uint32_t rank = cluster_rank();
  const int chunk = (total + S - 1) / S;
  const int e0 = static_cast<int>(rank) * chunk;
  const int e1 = min(total, e0 + chunk);
  const uint32_t base = smem_u32(part);
  for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += blockDim.x) {
    float v = 0.f;
    for (int q = 0; q < S; ++q) v += ld_dsmem_f32(map_smem_to_rank(base + 4u * static_cast<uint32_t>(e), q));
    store(e / BN, e % BN, v);
  }
  cluster_sync();  // keep this CTA's part alive until every peer has read it
}

}  // namespace wq
