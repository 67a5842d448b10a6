// wq_dequant.cu -- standalone dequantization of the packed weight formats into
// a dense [K, N] matrix in device memory: the separate-kernel path that the
// fused kernels are measured against.
//
// Definition ("融合反量化与GEMM：LLM推理的CUDA内核优化实践", 核心优化思路 and
// CUDA内核架构: the unfused path writes the dequantized weights to a buffer in
// DRAM and a separate GEMM reads them back; the per-weight formulas are those
// of the fused kernels):
//   W8:  w[k,n] = fp32(s[k/g, n] * q[k,n])                      (one rounding)
//   W3:  w[k,n] = fp16(fma(s[n], q(k,n), -zero[n]))             (fp32 fma, then fp16)
//   W4:  w[k,n] = act(s[g(k), n] * (q(k,n) - z[g(k), n]))       (exact in fp32, one rounding)
// with g(k) = g_idx[k] (act-order) or k / group.  Every kernel is a
// grid-stride loop over 16-byte loads of packed words (coalesced across n)
// and vector stores of dense rows; it is bound by HBM bandwidth.
#include "../../include/wq.h"
#include "wq_device.cuh"
#include "wq_launch.h"

namespace wq {

int device_sm_count();

namespace {

constexpr int kThreads = 256;

// Sign-extended byte b of a 32-bit word.
__device__ __forceinline__ int sbyte(uint32_t v, int b) { return static_cast<int32_t>(v << (24 - 8 * b)) >> 24; }

// 8-bit: one item = one row k, 16 consecutive columns (one 16-byte load of codes).
__global__ void __launch_bounds__(kThreads) dq8_kernel(const int8_t* __restrict__ w, const float* __restrict__ scales,
                                                       float* __restrict__ out, int K, int N, int group) {
  pdl_launch_dependents();
  pdl_wait();
  const int cpr = N / 16;
  const size_t items = size_t(K) * cpr;
  for (size_t i = size_t(blockIdx.x) * kThreads + threadIdx.x; i < items; i += size_t(gridDim.x) * kThreads) {
    const int k = static_cast<int>(i / cpr), n = static_cast<int>(i % cpr) * 16;
    const uint4 q = *reinterpret_cast<const uint4*>(w + size_t(k) * N + n);
    const float4* sp = reinterpret_cast<const float4*>(scales + size_t(k / group) * N + n);
    float4* op = reinterpret_cast<float4*>(out + size_t(k) * N + n);
    const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 s = sp[j];
      op[j] = make_float4(__fmul_rn(s.x, float(sbyte(qw[j], 0))), __fmul_rn(s.y, float(sbyte(qw[j], 1))),
                          __fmul_rn(s.z, float(sbyte(qw[j], 2))), __fmul_rn(s.w, float(sbyte(qw[j], 3))));
    }
  }
}

// 3-bit: one item = one 32-code block b (word rows 3b..3b+2), 4 consecutive
// columns.  Code j of a column is bits [3j, 3j+3) of the 96-bit little-endian
// stream w0 | w1 << 32 | w2 << 64.
__global__ void __launch_bounds__(kThreads) dq3_kernel(const int32_t* __restrict__ mat,
                                                       const uint16_t* __restrict__ scales,
                                                       const uint16_t* __restrict__ zeros, uint16_t* __restrict__ out,
                                                       int K, int N) {
  pdl_launch_dependents();
  pdl_wait();
  const int cpr = N / 4;
  const size_t items = size_t(K / 32) * cpr;
  for (size_t i = size_t(blockIdx.x) * kThreads + threadIdx.x; i < items; i += size_t(gridDim.x) * kThreads) {
    const int b = static_cast<int>(i / cpr), n = static_cast<int>(i % cpr) * 4;
    const uint4 a0 = *reinterpret_cast<const uint4*>(mat + size_t(3 * b) * N + n);
    const uint4 a1 = *reinterpret_cast<const uint4*>(mat + size_t(3 * b + 1) * N + n);
    const uint4 a2 = *reinterpret_cast<const uint4*>(mat + size_t(3 * b + 2) * N + n);
    const uint32_t w0[4] = {a0.x, a0.y, a0.z, a0.w}, w1[4] = {a1.x, a1.y, a1.z, a1.w},
                   w2[4] = {a2.x, a2.y, a2.z, a2.w};
    float s[4], nz[4];
    uint64_t lo[4], hi[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      s[c] = f16_bits_to_f32(scales[n + c]);
      nz[c] = -f16_bits_to_f32(zeros[n + c]);
      lo[c] = (uint64_t(w1[c]) << 32) | w0[c];
      hi[c] = (uint64_t(w2[c]) << 32) | w1[c];
    }
    uint16_t* op = out + size_t(32 * b) * N + n;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      uint32_t h[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t q = static_cast<uint32_t>((j < 21 ? lo[c] >> (3 * j) : hi[c] >> (3 * j - 32)) & 7u);
        h[c] = __half_as_ushort(__float2half_rn(fmaf(s[c], float(q), nz[c])));
      }
      *reinterpret_cast<uint2*>(op + size_t(j) * N) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    }
  }
}

// 4-bit: one item = one word row r (k = 8r..8r+7), 4 consecutive columns.
template <int ACT_BF16>
__global__ void __launch_bounds__(kThreads) dq4_kernel(const int32_t* __restrict__ qweight,
                                                       const uint16_t* __restrict__ scales,
                                                       const int32_t* __restrict__ qzeros,
                                                       const int32_t* __restrict__ g_idx, uint16_t* __restrict__ out,
                                                       int K, int N, int group) {
  pdl_launch_dependents();
  pdl_wait();
  const int G = K / group, cpr = N / 4;
  const size_t items = size_t(K / 8) * cpr;
  for (size_t i = size_t(blockIdx.x) * kThreads + threadIdx.x; i < items; i += size_t(gridDim.x) * kThreads) {
    const int r = static_cast<int>(i / cpr), n = static_cast<int>(i % cpr) * 4;
    const uint4 wv = *reinterpret_cast<const uint4*>(qweight + size_t(r) * N + n);
    const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = 8 * r + j;
      int g = g_idx ? g_idx[k] : k / group;
      g = min(max(g, 0), G - 1);  // out-of-range group ids are clamped, never read out of bounds
      const uint2 sb = *reinterpret_cast<const uint2*>(scales + size_t(g) * N + n);
      // zeros of columns n..n+3: four nibbles of one packed word (n % 8 is 0 or 4)
      const uint32_t zw = qzeros ? static_cast<uint32_t>(qzeros[size_t(g) * (N / 8) + n / 8]) >> (4 * (n % 8))
                                 : 0x8888u;
      const uint32_t sv[4] = {sb.x & 0xFFFFu, sb.x >> 16, sb.y & 0xFFFFu, sb.y >> 16};
      uint32_t h[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int q = static_cast<int>((w4[c] >> (4 * j)) & 15u) - static_cast<int>((zw >> (4 * c)) & 15u);
        // |q - z| <= 15 and the scale has at most 11 significant bits: the product is exact in fp32
        const float v = (ACT_BF16 ? bf16_bits_to_f32(sv[c]) : f16_bits_to_f32(sv[c])) * float(q);
        h[c] = f32_to_act<ACT_BF16>(v);
      }
      *reinterpret_cast<uint2*>(out + size_t(k) * N + n) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    }
  }
}

cudaError_t launch_simple(const void* kern, size_t items, unsigned flags, cudaStream_t stream, void** args) {
  const int n_sm = device_sm_count();
  const int sms = n_sm > 0 ? n_sm : 1;
  const size_t want = (items + kThreads - 1) / kThreads;
  const unsigned grid = static_cast<unsigned>(want < size_t(8) * sms ? (want > 0 ? want : 1) : size_t(8) * sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  if (flags & WQ_FLAG_PDL) {
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace

cudaError_t launch_wq8_dequant(const int8_t* w, const float* scales, float* out, int K, int N, int group,
                               unsigned flags, cudaStream_t stream) {
  void* args[] = {&w, &scales, &out, &K, &N, &group};
  return launch_simple(reinterpret_cast<const void*>(dq8_kernel), size_t(K) * (N / 16), flags, stream, args);
}

cudaError_t launch_wq3_dequant(const int32_t* mat, const void* scales, const void* zeros, void* out, int K, int N,
                               unsigned flags, cudaStream_t stream) {
  const uint16_t* s = static_cast<const uint16_t*>(scales);
  const uint16_t* z = static_cast<const uint16_t*>(zeros);
  uint16_t* o = static_cast<uint16_t*>(out);
  void* args[] = {&mat, &s, &z, &o, &K, &N};
  return launch_simple(reinterpret_cast<const void*>(dq3_kernel), size_t(K / 32) * (N / 4), flags, stream, args);
}

cudaError_t launch_wq4_dequant(const int32_t* qweight, const void* scales, const int32_t* qzeros,
                               const int32_t* g_idx, void* out, int K, int N, int group, int act_bf16,
                               unsigned flags, cudaStream_t stream) {
  const uint16_t* s = static_cast<const uint16_t*>(scales);
  uint16_t* o = static_cast<uint16_t*>(out);
  void* args[] = {&qweight, &s, &qzeros, &g_idx, &o, &K, &N, &group};
  const void* kern = act_bf16 ? reinterpret_cast<const void*>(dq4_kernel<1>)
                              : reinterpret_cast<const void*>(dq4_kernel<0>);
  return launch_simple(kern, size_t(K / 8) * (N / 4), flags, stream, args);
}

}  // namespace wq
