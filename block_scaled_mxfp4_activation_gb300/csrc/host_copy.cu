// Row copies between any two buffers the GPU can address, done by SM threads:
// the host-buffer entry (mxfp4_quant_gemm_host) moves a pinned, mapped host
// activation in through this (its result goes out from the GEMM kernel itself).
// On a GB300 node the GPU reaches host memory over the coherent NVLink-C2C
// link, and a small copy done by SM loads and stores finishes well before a DMA
// copy of the same size (which pays a fixed start-up latency of a few
// microseconds).
#include "internal.h"
#include "ptx.cuh"

namespace mxfp4 {

// Copies `rows` rows of `row_bytes` bytes (a multiple of 16; both pitches and
// both base addresses multiples of 16) from src to dst, 16 bytes per thread.
// Under programmatic launch the source is read into registers before the wait
// for the previous kernel when `src_early` is set (the source is not written
// by the stream's earlier kernels, e.g. host input), and every store comes
// after the wait (the destination may still be read by the previous kernel).
__global__ void __launch_bounds__(256) copy_rows_kernel(const uint8_t* __restrict__ src, int64_t src_pitch,
                                                        uint8_t* __restrict__ dst, int64_t dst_pitch,
                                                        int64_t row_bytes, int64_t rows, int src_early,
                                                        uint32_t* err) {
  grid_launch_dependents();
  const int64_t per_row = row_bytes / 16;
  const int64_t total = per_row * rows;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (src_early && i < total && i + stride >= total) {
    // one element per thread: load, then wait, then store
    const int64_t r = i / per_row, c = i - r * per_row;
    const bool ok = MXFP4_IN_BOUNDS(r < rows && c * 16 + 16 <= row_bytes, err);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (ok) v = *reinterpret_cast<const uint4*>(src + r * src_pitch + c * 16);
    grid_dependency_wait();
    if (ok) *reinterpret_cast<uint4*>(dst + r * dst_pitch + c * 16) = v;
    return;
  }
  grid_dependency_wait();
  for (; i < total; i += stride) {  // the source may be the previous grid's output
    const int64_t r = i / per_row, c = i - r * per_row;
    if (MXFP4_IN_BOUNDS(r < rows && c * 16 + 16 <= row_bytes, err))
      *reinterpret_cast<uint4*>(dst + r * dst_pitch + c * 16) = ld_after_wait_v4(src + r * src_pitch + c * 16);
  }
}

cudaError_t launch_copy_rows(const void* src, int64_t src_pitch, void* dst, int64_t dst_pitch, int64_t row_bytes,
                             int64_t rows, bool src_early, bool programmatic, int sm_count, cudaStream_t s) {
  const int64_t total = row_bytes / 16 * rows;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = 4 * static_cast<int64_t>(sm_count > 0 ? sm_count : 1);
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, copy_rows_kernel, static_cast<const uint8_t*>(src), src_pitch,
                            static_cast<uint8_t*>(dst), dst_pitch, row_bytes, rows, src_early ? 1 : 0,
                            device_error_word());
}

}  // namespace mxfp4
