/*
 * MXFP4 oracle: a plain, slow CPU statement of what the MXFP4 linear layer
 * computes.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the product library never does.
 * It shares no code, header or table with the CUDA path.
 *
 * Sources (the amd-mxfp4-mm leaderboard submissions on kernelindex.com):
 *   - submission 748756, `hw_pack_mxfp4`: block amax in fp32, the
 *     (bits + 0x200000) & 0xFF800000 power-of-two rounding, exponent - 129
 *     clamped to [-127, 127] and biased by 127 (the E8M0 byte).
 *   - submission 755056, "Software MXFP4 quant" (`_mxfp4_quant_tile`):
 *     q = x * 2^-s, rounded to E2M1 with round-to-nearest-even, saturating
 *     at 6, the sign OR'd in unconditionally, and two codes per byte with
 *     the even K index in the low nibble.
 *   - every submission's `tl.dot_scaled(..., "e2m1", ..., "e2m1", acc)`:
 *     C = sum_k deq(A)[m,k] * deq(B)[n,k], then cast to bf16.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - E2M1 rounding is "nearest representable magnitude, ties to the even
 *     code"; magnitudes above 6 give code 7 (6.0).
 *   - A negative input that rounds to zero keeps its sign (code 0x8).
 *   - The GEMM sums in fp64 in ascending k and rounds once, fp64 -> bf16,
 *     round-to-nearest-even.
 *   - B is quantized with the same rule as A.
 *
 * Everything is fp64 or integer; nothing here is blocked, fused or reordered.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* The eight E2M1 magnitudes, indexed by the 3-bit code (sign excluded). */
static const double kE2M1Magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

static uint32_t f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Magnitude of an E2M1 code (bit 3 = sign). */
double oracle_e2m1_decode(uint8_t code) {
  double v = kE2M1Magnitude[code & 7];
  return (code & 8) ? -v : v;
}

/* Value of an E8M0 byte: 2^(byte - 127).  Byte 0xFF (NaN) is never produced
 * by the quantizer; it decodes to NaN here. */
double oracle_e8m0_decode(uint8_t byte) {
  if (byte == 0xFF) return NAN;
  return ldexp(1.0, (int)byte - 127);
}

/* Encode |q| (an exact fp64 value) and a sign to an E2M1 code: the nearest of
 * the eight magnitudes, ties to the even code, anything above 6 -> code 7. */
uint8_t oracle_e2m1_encode(double q) {
  int neg = signbit(q) ? 1 : 0;
  double a = fabs(q);
  uint8_t best = 7;
  if (!(a > 6.0)) {
    double best_err = INFINITY;
    for (uint8_t c = 0; c < 8; ++c) {
      double err = fabs(a - kE2M1Magnitude[c]);
      if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
        best = c;
        best_err = err;
      }
    }
  }
  return (uint8_t)(best | (neg ? 8 : 0));
}

/* The block scale byte for a block whose largest magnitude is `amax`
 * (an fp32 value, as the pages compute it from bf16 inputs). */
uint8_t oracle_scale_byte(float amax) {
  uint32_t u = f32_bits(amax);
  u = (u + 0x200000u) & 0xFF800000u;
  int e = (int)((u >> 23) & 0xFF);
  int s = e - 129;
  if (s < -127) s = -127;
  if (s > 127) s = 127;
  return (uint8_t)(s + 127);
}

/* Quantize one row-major bf16 matrix x[rows, cols] (leading dimension ldx
 * elements; cols % 32 == 0) to packed E2M1 codes q[rows, cols/2] and E8M0
 * scales s[rows, cols/32], both dense row-major. */
void oracle_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                     uint8_t* s) {
  const int64_t nblk = cols / 32;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nblk; ++b) {
      const uint16_t* blk = x + r * ldx + b * 32;
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) {
        float a = fabsf(bf16_to_f32(blk[i]));
        if (a > amax) amax = a;
      }
      uint8_t sb = oracle_scale_byte(amax);
      s[r * nblk + b] = sb;
      int sexp = (int)sb - 127;
      uint8_t codes[32];
      for (int i = 0; i < 32; ++i) {
        double v = (double)bf16_to_f32(blk[i]);
        codes[i] = oracle_e2m1_encode(ldexp(v, -sexp));
      }
      for (int i = 0; i < 16; ++i) {
        q[r * (cols / 2) + b * 16 + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
      }
    }
  }
}

/* Dequantize packed codes + scales back to fp64 values x[rows, cols]. */
void oracle_dequantize(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t cols, double* x) {
  const int64_t nblk = cols / 32;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t k = 0; k < cols; ++k) {
      uint8_t byte = q[r * (cols / 2) + k / 2];
      uint8_t code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      x[r * cols + k] = oracle_e2m1_decode(code) * oracle_e8m0_decode(s[r * nblk + k / 32]);
    }
  }
}

/* Round an fp64 value to bf16, round-to-nearest-even, in one step.
 * bf16 has 8 significant bits and a minimum exponent of -126 (subnormal
 * quantum 2^-133); |results| at or above 2^128 overflow to infinity. */
uint16_t oracle_bf16_from_f64(double d) {
  if (isnan(d)) return 0x7FC0;
  double r;
  if (d == 0.0 || isinf(d)) {
    r = d;
  } else {
    int e;
    frexp(d, &e); /* d = m * 2^e, 0.5 <= |m| < 1 */
    int quantum = e - 8;
    if (quantum < -133) quantum = -133;
    r = ldexp(nearbyint(ldexp(d, -quantum)), quantum); /* default mode: ties to even */
    if (fabs(r) >= ldexp(1.0, 128)) r = copysign(INFINITY, d);
  }
  /* r is exactly representable in bf16 (or is +-0 / +-inf): narrow via fp32. */
  float f = (float)r;
  return (uint16_t)(f32_bits(f) >> 16);
}

/* C[m, n] = sum_k A[m, k] * B[n, k] over dequantized operands, fp64, ascending k.
 * Writes the fp64 sums to c64 (if non-null) and their bf16 rounding to c16. */
void oracle_gemm(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs,
                 int64_t M, int64_t N, int64_t K, double* c64, uint16_t* c16) {
  const int64_t kh = K / 2, nblk = K / 32;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        uint8_t ab = aq[m * kh + k / 2], bb = bq[n * kh + k / 2];
        uint8_t ac = (k % 2 == 0) ? (ab & 0xF) : (ab >> 4);
        uint8_t bc = (k % 2 == 0) ? (bb & 0xF) : (bb >> 4);
        double va = oracle_e2m1_decode(ac) * oracle_e8m0_decode(as[m * nblk + k / 32]);
        double vb = oracle_e2m1_decode(bc) * oracle_e8m0_decode(bs[n * nblk + k / 32]);
        acc += va * vb;
      }
      if (c64) c64[m * N + n] = acc;
      if (c16) c16[m * N + n] = oracle_bf16_from_f64(acc);
    }
  }
}

/* The same sum for an explicit list of (m, n) output positions; used to check
 * large outputs element by element on a sample. */
void oracle_gemm_sampled(const uint8_t* aq, const uint8_t* as, const uint8_t* bq,
                         const uint8_t* bs, int64_t K, const int64_t* ms, const int64_t* ns,
                         int64_t count, double* c64, uint16_t* c16) {
  const int64_t kh = K / 2, nblk = K / 32;
  for (int64_t i = 0; i < count; ++i) {
    const uint8_t* ar = aq + ms[i] * kh;
    const uint8_t* br = bq + ns[i] * kh;
    const uint8_t* asr = as + ms[i] * nblk;
    const uint8_t* bsr = bs + ns[i] * nblk;
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      uint8_t ac = (k % 2 == 0) ? (ar[k / 2] & 0xF) : (ar[k / 2] >> 4);
      uint8_t bc = (k % 2 == 0) ? (br[k / 2] & 0xF) : (br[k / 2] >> 4);
      acc += (oracle_e2m1_decode(ac) * oracle_e8m0_decode(asr[k / 32])) *
             (oracle_e2m1_decode(bc) * oracle_e8m0_decode(bsr[k / 32]));
    }
    if (c64) c64[i] = acc;
    if (c16) c16[i] = oracle_bf16_from_f64(acc);
  }
}

/* The whole linear layer: quantize the bf16 activation a[M, K] (leading
 * dimension lda) with the rule above, then multiply by the pre-quantized
 * weight (bq, bs) and round to bf16.  aq/as receive the activation codes. */
void oracle_quant_gemm(const uint16_t* a, int64_t lda, const uint8_t* bq, const uint8_t* bs,
                       int64_t M, int64_t N, int64_t K, uint8_t* aq, uint8_t* as, double* c64,
                       uint16_t* c16) {
  oracle_quantize(a, M, K, lda, aq, as);
  oracle_gemm(aq, as, bq, bs, M, N, K, c64, c16);
}

/* Element-wise array forms of the scalar rules above, for the tests. */
void oracle_e2m1_encode_array(const double* q, int64_t n, uint8_t* codes) {
  for (int64_t i = 0; i < n; ++i) codes[i] = oracle_e2m1_encode(q[i]);
}

void oracle_scale_byte_array(const float* amax, int64_t n, uint8_t* bytes) {
  for (int64_t i = 0; i < n; ++i) bytes[i] = oracle_scale_byte(amax[i]);
}

void oracle_bf16_from_f64_array(const double* d, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_from_f64(d[i]);
}
