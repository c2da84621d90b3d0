// MXFP4 block quantization arithmetic shared by the standalone quantize kernel
// and the fused GEMM's activation producer: in both, two adjacent lanes own
// one 32-element block, 16 bf16 values each, and combine their maxima with
// one shuffle.
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

// E8M0 byte of a block from its amax (bf16 bit pattern).
__device__ __forceinline__ uint32_t scale_byte_from_amax(uint32_t amax_bf16) {
  const uint32_t u = ((amax_bf16 << 16) + 0x200000u) & 0xFF800000u;
  int s = static_cast<int>(u >> 23) - 129;
  s = max(-127, min(127, s));
  return static_cast<uint32_t>(s + 127);
}

// Largest |x| of 16 bf16 values (two 16-byte words), as a bf16 bit pattern
// (sign cleared).  Works on the integer patterns: for non-negative finite
// floats the integer order is the numeric order, and nothing is flushed to
// zero.
__device__ __forceinline__ uint32_t absmax16_bf16(uint4 v, uint4 w) {
  const uint32_t m = 0x7FFF7FFFu;
  uint32_t a = __vmaxu2(v.x & m, v.y & m);
  uint32_t b = __vmaxu2(v.z & m, v.w & m);
  a = __vmaxu2(a, __vmaxu2(w.x & m, w.y & m));
  b = __vmaxu2(b, __vmaxu2(w.z & m, w.w & m));
  a = __vmaxu2(a, b);
  return max(a & 0xFFFFu, a >> 16);
}

// 2^-s for scale byte s + 127, as a bf16 bit pattern: a normal number for
// every byte a finite input produces (0..253).
__device__ __forceinline__ uint16_t scale_bf16_from_byte(uint32_t byte) {
  return static_cast<uint16_t>((254u - byte) << 7);
}

// 8 bf16 values (one 16-byte word, element i in half i of the vector) times
// 2^-s -> 8 E2M1 codes in 4 bytes, element 2i in the low nibble of byte i.
// The product is formed by mixed-precision FMAs straight from the bf16 halves
// (bf16 x bf16 + fp32 -> fp32): x * 2^-s is exact in fp32 whenever it matters
// (its magnitude is at least 2^-126 or the code is 0 either way), and the
// addend -0 leaves every product unchanged, including the sign of a zero.
// The four code bytes are gathered into one 32-bit word directly.
__device__ __forceinline__ uint32_t e2m1_pack8(uint4 v, uint16_t scale_bf16) {
  uint32_t out;
  asm("{\n\t.reg .b16 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
      ".reg .f32 y0, y1, y2, y3, y4, y5, y6, y7;\n\t"
      ".reg .b8 c0, c1, c2, c3;\n\t"
      "mov.b32 {l0, h0}, %1;\n\t"
      "mov.b32 {l1, h1}, %2;\n\t"
      "mov.b32 {l2, h2}, %3;\n\t"
      "mov.b32 {l3, h3}, %4;\n\t"
      "fma.rn.f32.bf16 y0, l0, %5, 0f80000000;\n\t"
      "fma.rn.f32.bf16 y1, h0, %5, 0f80000000;\n\t"
      "fma.rn.f32.bf16 y2, l1, %5, 0f80000000;\n\t"
      "fma.rn.f32.bf16 y3, h1, %5, 0f80000000;\n\t"
      "fma.rn.f32.bf16 y4, l2, %5, 0f80000000;\n\t"
      "fma.rn.f32.bf16 y5, h2, %5, 0f80000000;\n\t"
      "fma.rn.f32.bf16 y6, l3, %5, 0f80000000;\n\t"
      "fma.rn.f32.bf16 y7, h3, %5, 0f80000000;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c0, y1, y0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c1, y3, y2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c2, y5, y4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c3, y7, y6;\n\t"
      "mov.b32 %0, {c0, c1, c2, c3};\n\t}"
      : "=r"(out)
      : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "h"(scale_bf16));
  return out;
}

// Two bf16 values (pair: element 2i in the low half, 2i + 1 in the high half)
// times 2^-s -> one byte of two E2M1 codes, element 2i in the low nibble: the
// same instructions as e2m1_pack8, for one pair.
__device__ __forceinline__ uint32_t e2m1_pack2(uint32_t pair, uint16_t scale_bf16) {
  uint32_t out;
  asm("{\n\t.reg .b16 l0, h0;\n\t"
      ".reg .f32 y0, y1;\n\t"
      ".reg .b8 c0;\n\t"
      "mov.b32 {l0, h0}, %1;\n\t"
      "fma.rn.f32.bf16 y0, l0, %2, 0f80000000;\n\t"
      "fma.rn.f32.bf16 y1, h0, %2, 0f80000000;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c0, y1, y0;\n\t"
      "cvt.u32.u8 %0, c0;\n\t}"
      : "=r"(out)
      : "r"(pair), "h"(scale_bf16));
  return out;
}

}  // namespace mxfp4
