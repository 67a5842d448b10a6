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

}  // namespace

int actorder_prepare(const int32_t* qweight, const int32_t* g_idx, int K, int N, int group, int32_t* qweight_sorted,
                     int32_t* perm, cudaStream_t stream) {
  const int G = K / group;
  std::vector<int32_t> gi(K), p(K);
  if (cudaMemcpyAsync(gi.data(), g_idx, sizeof(int32_t) * K, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return 2;
  // counting sort by group, stable in k; every group must hold exactly `group` rows
  std::vector<int> count(G, 0);
  for (int k = 0; k < K; ++k) {
    if (gi[k] < 0 || gi[k] >= G) return 1;
    ++count[gi[k]];
  }
  for (int g = 0; g < G; ++g)
    if (count[g] != group) return 1;
  std::vector<int> next(G);
  for (int g = 0; g < G; ++g) next[g] = g * group;
  for (int k = 0; k < K; ++k) p[next[gi[k]]++] = k;
  if (cudaMemcpyAsync(perm, p.data(), sizeof(int32_t) * K, cudaMemcpyHostToDevice, stream) != cudaSuccess) return 2;
  dim3 grid((N + 255) / 256, K / 8);
  repack_sorted_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(qweight), perm, K, N,
                                                  reinterpret_cast<uint32_t*>(qweight_sorted));
  if (cudaGetLastError() != cudaSuccess) return 2;
  return cudaStreamSynchronize(stream) == cudaSuccess ? 0 : 2;  // the host vectors go out of scope
}

}  // namespace wq
