// MXFP4 block quantization arithmetic shared by the standalone quantize kernel
// and the fused GEMM's activation producer.  One thread owns 8 consecutive
// bf16 values (16 bytes); four adjacent lanes own one 32-element block and
// combine their maxima with two butterfly shuffles.
//
// Rule (amd-mxfp4-mm submission 748756, `hw_pack_mxfp4`; submission 755056,
// "Software MXFP4 quant"): amax = max |x| over the block; u = (bits(amax) +
// 0x200000) & 0xFF800000; s = clamp(exponent field of u - 129, -127, 127);
// scale byte = s + 127; code = E2M1(x * 2^-s), round to nearest even,
// saturating at 6, sign kept; two codes per byte, even index low.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace mxfp4 {

// Largest |x| of 8 bf16 values, as a bf16 bit pattern (sign cleared).  Works
// on the integer patterns: for non-negative finite floats the integer order
// is the numeric order, and nothing is flushed to zero.
__device__ __forceinline__ uint32_t absmax8_bf16(uint4 v) {
  const uint32_t m = 0x7FFF7FFFu;
  uint32_t a = __vmaxu2(v.x & m, v.y & m);
  uint32_t b = __vmaxu2(v.z & m, v.w & m);
  a = __vmaxu2(a, b);
  return max(a & 0xFFFFu, a >> 16);
}

// E8M0 byte of a block from its amax (bf16 bit pattern).
__device__ __forceinline__ uint32_t scale_byte_from_amax(uint32_t amax_bf16) {
  const uint32_t u = ((amax_bf16 << 16) + 0x200000u) & 0xFF800000u;
  int s = static_cast<int>(u >> 23) - 129;
  s = max(-127, min(127, s));
  return static_cast<uint32_t>(s + 127);
}

// 2^-s for scale byte s + 127; a normal fp32 for every byte a finite input
// produces (0..253).
__device__ __forceinline__ float inv_scale_from_byte(uint32_t byte) {
  return __uint_as_float((254u - byte) << 23);
}

// 8 bf16 values (one 16-byte word, element i in half i of the vector) times
// 2^-s -> 8 E2M1 codes in 4 bytes, element 2i in the low nibble of byte i.
// x * 2^-s is exact in fp32 whenever it matters (its magnitude is at least
// 2^-126 or the code is 0 either way), and __fmul_rn keeps subnormal inputs.
__device__ __forceinline__ uint32_t e2m1_pack8(uint4 v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __fmul_rn(__uint_as_float(w[i] << 16), inv);
    const float hi = __fmul_rn(__uint_as_float(w[i] & 0xFFFF0000u), inv);
    out |= cvt_e2m1x2(hi, lo) << (8 * i);
  }
  return out;
}

// Quantizes the 8 values a lane owns as part of a 32-element block spread over
// the 4 lanes lane^1, lane^2, lane^3 (all 32 lanes must call it together).
// Returns the 4 code bytes; *byte_out receives the block's scale byte.
__device__ __forceinline__ uint32_t quantize_quad(uint4 v, uint32_t* byte_out) {
  uint32_t amax = absmax8_bf16(v);
  amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  const uint32_t byte = scale_byte_from_amax(amax);
  *byte_out = byte;
  return e2m1_pack8(v, inv_scale_from_byte(byte));
}

}  // namespace mxfp4
