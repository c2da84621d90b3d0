// The fused layer's two-pass route (quantize A into scratch, then the GEMM on
// the codes) with its scratch in a fixed device array that the library owns,
// for callers that cannot allocate device memory: a plugin running inside a
// host framework that reserves all device memory up front and forbids
// allocation afterwards, or code that must not call cudaMalloc because it
// synchronises the device.  The caller passes only inputs and outputs.
//
// Every GPU that loads the library holds this array (kStaticScratchBytes)
// until the process exits.  All calls share it, so calls that can overlap on
// the GPU (different streams without ordering between them) race on it.
#include <mutex>

#include "internal.h"

namespace mxfp4 {
namespace {

// 4 MiB: room for the codes and scales of an activation of up to ~7.9 M
// elements (for example M = 1024, K = 7168).
constexpr size_t kStaticScratchBytes = size_t(4) << 20;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// The array's device address on the current device.  In host code the name
// g_static_scratch is only a host-side stand-in, so the address is looked up
// once per device with that device current, and the result checked.
uint8_t* static_scratch_address(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  static std::mutex mu;
  static uint8_t* addr[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_static_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = static_cast<uint8_t*>(p);
  }
  *err = cudaSuccess;
  return addr[dev];
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace mxfp4

using namespace mxfp4;

extern "C" mxfp4_status_t mxfp4_quant_gemm_static_scratch(const void* A, int64_t lda, const void* Bpacked,
                                                          void* C, int64_t M, int64_t N, int64_t K,
                                                          mxfp4_stream_t stream) {
  // The size limits of the GEMM entries, then this entry's own limit, then
  // pointers, the device and the array's address; two_pass() makes every
  // remaining check of both launches (plan and tensor maps included) before
  // the first one, so a call that returns an error has launched nothing.
  mxfp4_status_t st = check_mnk(M, N, K);
  if (st != MXFP4_OK) return st;
  if (A == nullptr || Bpacked == nullptr || C == nullptr || lda < K) return MXFP4_ERR_INVALID_ARG;
  const size_t codes = round256(static_cast<size_t>(M) * static_cast<size_t>(K / 2));
  const size_t need = codes + round256(static_cast<size_t>(M) * static_cast<size_t>(K / 32));
  if (need > kStaticScratchBytes) {
    set_last_error("the activation's codes and scales exceed the library's static scratch (4 MiB)");
    return MXFP4_ERR_UNSUPPORTED_SHAPE;
  }
  const uintptr_t mis = reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(Bpacked) |
                        reinterpret_cast<uintptr_t>(C);
  if ((mis & 15u) != 0 || lda % 8 != 0) return MXFP4_ERR_MISALIGNED;
  st = check_device();
  if (st != MXFP4_OK) return st;
  cudaError_t e;
  uint8_t* scratch = static_scratch_address(&e);
  if (scratch == nullptr) {
    set_last_error(e == cudaSuccess ? "no device address for the static scratch" : cudaGetErrorString(e));
    return MXFP4_ERR_CUDA;
  }
  // Quantization overwrites every byte the GEMM then reads, so nothing needs
  // clearing between calls.
  return two_pass(A, lda, Bpacked, C, M, N, K, scratch, scratch + codes, reinterpret_cast<cudaStream_t>(stream),
                  nullptr);
}
