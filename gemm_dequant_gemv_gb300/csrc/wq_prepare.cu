// wq_prepare.cu -- one-time preparation of act-order 4-bit weights: the rows
// are sorted by their group (stable in k), so that each group becomes a
// contiguous run of `group` rows and the GEMV can apply one scale per group
// instead of gathering a scale per code.  Sorted row i holds original row
// perm[i]; the product is unchanged because x is read through the same perm.
#include <cuda_runtime.h>

#include <vector>

#include "wq_mma.h"

namespace wq {
namespace {

// qs[r', n] nibble j = code of original row perm[8 r' + j] in column n.
__global__ void repack_sorted_kernel(const uint32_t* __restrict__ qw, const int32_t* __restrict__ perm, int K, int N,
                                     uint32_t* __restrict__ qs) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int r = blockIdx.y;
  if (n >= N) return;
  uint32_t w = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    int k = perm[8 * r + j];
    k = min(max(k, 0), K - 1);
    const uint32_t src = qw[size_t(k / 8) * N + n];
    w |= ((src >> (4 * (k % 8))) & 15u) << (4 * j);
  }
  qs[size_t(r) * N + n] = w;
}

// The tiled layout of the tensor-core GEMV (wq_gemv4t.cu): word (r, n) of the
// GPTQ matrix (rows sorted through perm when perm != null) goes to
//   ((r/8 * (N/32) + slab) * 256) + ((r%8) % 2) * 128 + (4 g + (r%8) / 2) * 4 + i,
// slab = n / 32, g = (n % 32) / 4, i = n % 4: every 64-value unit of a 32-column
// slab is one contiguous 1 KB block, in which the 16 bytes thread (g, t) reads
// for word row 2t + ab sit at offset ab * 512 + (4g + t) * 16; the blocks of
// one unit are contiguous over the slabs, so a CTA's columns of one unit are
// one copy, and the CTAs streaming at the same time read neighbouring blocks.
__global__ void repack_tiled_kernel(const uint32_t* __restrict__ qw, const int32_t* __restrict__ perm, int K, int N,
                                    uint32_t* __restrict__ out) {
  const size_t o = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t total = size_t(K / 8) * N;
  if (o >= total) return;
  const int i = int(o & 3u), lane = int((o >> 2) & 31u), ab = int((o >> 7) & 1u);
  const size_t blk = o >> 8;  // unit * (N / 32) + slab
  const int unit = int(blk / (N / 32)), slab = int(blk % (N / 32));
  const int g = lane >> 2, t = lane & 3;
  const int r = 8 * unit + 2 * t + ab, n = 32 * slab + 4 * g + i;
  uint32_t w;
  if (perm) {
    w = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      int k = perm[8 * r + j];
      k = min(max(k, 0), K - 1);
      const uint32_t src = qw[size_t(k / 8) * N + n];
      w |= ((src >> (4 * (k % 8))) & 15u) << (4 * j);
    }
  } else {
    w = qw[size_t(r) * N + n];
  }
  out[o] = w;
}

// Counting sort of the rows by group, stable in k: p[i] = original row of
// sorted row i.  Returns false unless every group holds exactly `group` rows.
bool sort_by_group(const std::vector<int32_t>& gi, int K, int group, std::vector<int32_t>& p) {
  const int G = K / group;
  std::vector<int> count(G, 0);
  for (int k = 0; k < K; ++k) {
    if (gi[k] < 0 || gi[k] >= G) return false;
    ++count[gi[k]];
  }
  for (int g = 0; g < G; ++g)
    if (count[g] != group) return false;
  std::vector<int> next(G);
  for (int g = 0; g < G; ++g) next[g] = g * group;
  p.assign(K, 0);
  for (int k = 0; k < K; ++k) p[next[gi[k]]++] = k;
  return true;
}

}  // namespace

int repack_tiled(const int32_t* qweight, const int32_t* g_idx, int K, int N, int group, int32_t* qweight_tiled,
                 int32_t* perm, cudaStream_t stream) {
  if (g_idx) {
    std::vector<int32_t> gi(K), p;
    if (cudaMemcpyAsync(gi.data(), g_idx, sizeof(int32_t) * K, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
      return 2;
    if (!sort_by_group(gi, K, group, p)) return 1;
    if (cudaMemcpyAsync(perm, p.data(), sizeof(int32_t) * K, cudaMemcpyHostToDevice, stream) != cudaSuccess) return 2;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return 2;  // p goes out of scope
  }
  const size_t total = size_t(K / 8) * N;
  repack_tiled_kernel<<<unsigned((total + 255) / 256), 256, 0, stream>>>(
      reinterpret_cast<const uint32_t*>(qweight), g_idx ? perm : nullptr, K, N, reinterpret_cast<uint32_t*>(qweight_tiled));
  if (cudaGetLastError() != cudaSuccess) return 2;
  return cudaStreamSynchronize(stream) == cudaSuccess ? 0 : 2;
}

int actorder_prepare(const int32_t* qweight, const int32_t* g_idx, int K, int N, int group, int32_t* qweight_sorted,
                     int32_t* perm, cudaStream_t stream) {
  std::vector<int32_t> gi(K), p;
  if (cudaMemcpyAsync(gi.data(), g_idx, sizeof(int32_t) * K, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return 2;
  if (!sort_by_group(gi, K, group, p)) return 1;  // every group must hold exactly `group` rows
  if (cudaMemcpyAsync(perm, p.data(), sizeof(int32_t) * K, cudaMemcpyHostToDevice, stream) != cudaSuccess) return 2;
  dim3 grid((N + 255) / 256, K / 8);
  repack_sorted_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(qweight), perm, K, N,
                                                  reinterpret_cast<uint32_t*>(qweight_sorted));
  if (cudaGetLastError() != cudaSuccess) return 2;
  return cudaStreamSynchronize(stream) == cudaSuccess ? 0 : 2;  // the host vectors go out of scope
}

}  // namespace wq
