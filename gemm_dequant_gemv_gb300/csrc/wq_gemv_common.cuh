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
//   * warps 0..7 are consumers: per stage they first convert the stage's x
//     block cooperatively (one named barrier), then each takes one "unit" (a
//     fixed number of packed rows), unpacks the codes in registers, converts
//     them with exact bit tricks and accumulates in fp32 with packed FFMA2.
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

// Final reduction of the S partial tiles of a cluster and the store of y.
// `part` is this CTA's [MT][BN] fp32 partial in shared memory, written by the
// consumer warps.  Every thread of the CTA must call this (it contains CTA-
// and cluster-wide barriers).  The S CTAs of a cluster each reduce one
// contiguous chunk of the tile, reading the other CTAs' partials through
// distributed shared memory in rank order (a fixed summation order: the
// result does not depend on timing).  store(m, col, value) writes one output.
template <int MT, int BN, class StoreFn>
__device__ __forceinline__ void finish_tile(const float* part, int S, StoreFn store) {
  constexpr int total = MT * BN;
  if (S == 1) {
    __syncthreads();
    for (int e = threadIdx.x; e < total; e += blockDim.x) store(e / BN, e % BN, part[e]);
    return;
  }
  cluster_sync();
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int chunk = (total + S - 1) / S;
  const int e0 = static_cast<int>(rank) * chunk;
  const int e1 = min(total, e0 + chunk);
  const uint32_t base = smem_u32(part);
  for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += blockDim.x) {
    float v = 0.f;
    for (int q = 0; q < S; ++q) v += ld_dsmem_f32(map_smem_to_rank(base + 4u * static_cast<uint32_t>(e), q));
    store(e / BN, e % BN, v);
  }
  cluster_sync();
}

}  // namespace wq
