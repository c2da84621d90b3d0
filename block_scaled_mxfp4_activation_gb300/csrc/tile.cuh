// Geometry of the block-scaled tcgen05 MMA shared by the GEMM kernels: the
// instruction descriptor and the byte layout of a tensor-memory scale chunk.
#pragma once

#include <cstdint>

#include "internal.h"

namespace mxfp4 {

// Instruction descriptor of kind::mxf4 (E2M1 x E2M1, UE8M0 scales, fp32
// accumulate): A/B formats at bits 7-9 / 10-12 (E2M1 = 1), both K-major, N >> 3
// at bits 17-22, scale type UE8M0 at bit 23, M >> 4 at bits 24-28; the byte of
// each scale word used by this MMA (0 or 2: scales 0-1 or 2-3 of a 4-scale
// chunk) at bits 29-30 (A) and 4-5 (B).
template <int BM>
__device__ __forceinline__ uint32_t mxf4_idesc(uint32_t scale_id) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BM >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(kTileN >> 4) << 24) | (scale_id << 29) | (scale_id << 4);
}

// Byte offset of scale j (0..3) of row r in a 128-row x 4-scale chunk.
__device__ __forceinline__ uint32_t sf_chunk_offset(int r) { return (r & 31) * 16 + ((r & 127) >> 5) * 4; }

}  // namespace mxfp4
