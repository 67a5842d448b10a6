// w8a8_noalloc.cu -- w8a8_gemm for callers that cannot allocate device memory.
//
// The W8A8 path needs device scratch between its two kernels (the fp16 copies
// of the quantized activations and the row scales).  w8a8_gemm takes that
// scratch from the caller; w8a8_gemm_noalloc instead uses a fixed-size array
// compiled into the library, so the call allocates nothing.  The computation
// is w8a8_gemm's, unchanged: this file only supplies the scratch pointer.
#include <stdint.h>

#include <mutex>

#include "../../include/wq.h"

namespace wq {
namespace {

// Largest scratch the built-in array offers: 8 MiB.  w8a8_gemm needs
// align256(2*M*K) + align256(4*M) bytes, so for example M <= 511 at K = 8192
// or M <= 1023 at K = 4096 (M = 512 at K = 8192 needs 8 MiB + 2048 bytes).
constexpr size_t kScratchBytes = size_t(8) << 20;

// The scratch itself, one copy per device (module-scope device memory).
// Nothing in it needs to start at zero: every call writes each byte it later
// reads.
static __device__ __align__(256) unsigned char g_w8a8_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};  // device address of g_w8a8_scratch, per device ordinal

// The device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.  In host code the array's
// name only stands in for the symbol; the address comes from the runtime.
cudaError_t scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_w8a8_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace wq

extern "C" {

WQ_API size_t w8a8_gemm_noalloc_max_scratch_bytes(void) { return wq::kScratchBytes; }

WQ_API wq_status w8a8_gemm_noalloc(const void* X, const int8_t* W, const float* Sw, void* Y, int M, int K, int N,
                                   int8_t* Xq_out, float* Sx_out, int32_t* acc_out, unsigned flags,
                                   void* stream) {
  // the checks w8a8_gemm makes, repeated here so that a bad call touches no CUDA state
  if (!X || !W || !Sw || !Y) return WQ_ERR_NULL;
  if (M < 1 || K < 64 || N < 16 || K > 65536 || K % 64 != 0 || N % 16 != 0) return WQ_ERR_SHAPE;
  if (!wq::aligned16(X) || !wq::aligned16(W) || !wq::aligned16(Sw) || !wq::aligned16(Y) ||
      (Xq_out && !wq::aligned16(Xq_out)) || (Sx_out && !wq::aligned16(Sx_out)) ||
      (acc_out && !wq::aligned16(acc_out)))
    return WQ_ERR_ALIGN;
  const size_t need = w8a8_gemm_workspace_bytes(M, K, N);
  if (need == 0) return WQ_ERR_SHAPE;
  if (need > wq::kScratchBytes) return WQ_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (wq::scratch_on_current_device(&scratch) != cudaSuccess) return WQ_ERR_CUDA;
  return w8a8_gemm(X, W, Sw, Y, M, K, N, Xq_out, Sx_out, acc_out, scratch, wq::kScratchBytes, flags, stream);
}

}  // extern "C"
