// NVFP4 encoding on the device: 16-element blocks along K, E2M1 nibbles
// (low nibble = even K index), one FP8-E4M3 block scale per block, under an
// FP32 global scale gs that is multiplied into x.
//
// Rules (nvfp4-megamoe-kernel commit pages, cutedsl/bridge.py page,
// "Bug #3 fix" and "Bug #4 fix" paragraphs):
//   x' = x * gs (FP32), b = max |x'| over the block,
//   b < 6 * 2^-9  -> scale 0 and all 16 nibbles 0 (zero and underflow blocks),
//   else scale = E4M3(b / 6) (IEEE division, round to nearest even, saturating),
//        q = x' / dec(scale) (IEEE division), nibble = E2M1(q) (nearest, ties to even,
//        saturating at 6); a magnitude that rounds to 0 carries no sign.
// Scales are stored in the 128-row x 4-column tile layout read by the
// block-scaled MMA: see sf_offset().
#pragma once
#include <cstdint>

namespace nvfp4 {

constexpr float kUnderflowAmax = 0.01171875f;  // 6 * 2^-9, exact in FP32
constexpr float kGsNumerator = 2688.0f;        // 448 * 6

// Byte offset of scale (row r, scale column c) in a buffer with `cols4`
// scale columns (a multiple of 4): 512-byte tiles of 128 rows x 4 columns,
// tiles ordered along the columns first; inside a tile the 16-byte line
// r%32 holds rows r%32, +32, +64, +96 (4 bytes each, one per column).
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t cols4) {
  return (((r >> 7) * (cols4 >> 2) + (c >> 2)) << 9) + ((r & 31) << 4) + (((r & 127) >> 5) << 2) + (c & 3);
}

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xFu, m = code & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
}

// Round-to-nearest-even, saturating FP32 -> E4M3 (PTX cvt, both halves from one value).
__device__ __forceinline__ uint32_t e4m3_code(float v) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(d) : "f"(v));
  return d & 0xFFu;
}

// Two E2M1 codes in one byte: `lo` -> bits 0-3, `hi` -> bits 4-7 (round to
// nearest even, saturating at 6).  The PTX cvt puts its first source operand
// in the upper half of the result.
__device__ __forceinline__ uint32_t e2m1x2_code(float lo, float hi) {
  uint32_t r;
  asm("{\n.reg .b8 t;\ncvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\ncvt.u32.u8 %0, t;\n}" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight E2M1 codes in one word: element 2j in the low nibble of byte j
// (four paired conversions into byte registers, packed by one move).
__device__ __forceinline__ uint32_t e2m1x8_word(float q0, float q1, float q2, float q3, float q4, float q5, float q6,
                                                float q7) {
  uint32_t w;
  asm("{\n.reg .b8 b0, b1, b2, b3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      "mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(w)
      : "f"(q0), "f"(q1), "f"(q2), "f"(q3), "f"(q4), "f"(q5), "f"(q6), "f"(q7));
  return w;
}

// Clear the sign bit of every nibble whose magnitude bits are zero (-0 -> 0).
__device__ __forceinline__ uint32_t drop_negative_zero(uint32_t w) {
  const uint32_t mag = w & 0x77777777u;
  const uint32_t nonzero = (mag + 0x77777777u) & 0x88888888u;
  return mag | (w & nonzero);
}

// x / d rounded to nearest even, for a block scale d and y = RN(1/d):
// q0 = RN(x*y) is within one ulp of x/d, the remainder x - q0*d is exact
// with a fused multiply-add, and one correction step q0 + r*y rounds to the
// correctly rounded quotient (Markstein's theorem for a correctly rounded
// reciprocal).  Equality with the IEEE division is checked exhaustively on
// the device by the test-suite for every E4M3 scale value.
__device__ __forceinline__ float div_by_scale(float x, float d, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r = __fmaf_rn(-q0, d, x);
  return __fmaf_rn(r, y, q0);
}

// Packed pairs of FP32 values (element 2j in the low half, 2j+1 in the high
// half), each half rounded exactly like its scalar operation.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Quantize one block of 16 already globally-scaled values given as 8 packed
// pairs, with the block maximum b given.  Returns the scale code; writes 8
// packed bytes (element 2j in the low nibble of byte j).  b / 6 and every
// x' / dec(scale) are the correctly rounded quotients (div_by_scale; 6 is an
// E4M3 value; rcp6 = RN(1/6)), two elements per instruction where possible.
__device__ __forceinline__ uint32_t quant_block16_pairs(const uint64_t (&xs2)[8], float b, float rcp6, uint32_t& lo,
                                                        uint32_t& hi) {
  lo = hi = 0u;
  if (!(b >= kUnderflowAmax)) return 0u;
  const uint32_t s = e4m3_code(div_by_scale(fminf(b, 3.40282347e38f), 6.0f, rcp6));
  const float d = e4m3_value(s);
  const float y = __frcp_rn(d);
  const uint64_t y2 = f2_pack(y, y), nd2 = f2_pack(-d, -d);
  float q[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint64_t q0 = f2_mul(xs2[j], y2);
    const uint64_t r = f2_fma(q0, nd2, xs2[j]);
    f2_unpack(f2_fma(r, y2, q0), q[2 * j], q[2 * j + 1]);
  }
  lo = drop_negative_zero(e2m1x8_word(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]));
  hi = drop_negative_zero(e2m1x8_word(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]));
  return s;
}

// FP8 block form of the L1 output: E4M3 codes in blocks of 16 values with a
// power-of-two scale 2^k, k the least integer with amax <= 448 * 2^k
// (448 = 1.75 * 2^8: with amax = m * 2^E, k = E - 8, plus 1 when m > 1.75),
// clamped to [-126, 126]; 0 for an all-zero block.
__device__ __forceinline__ int fp8_block_k(float amax) {
  const uint32_t b = __float_as_uint(amax);
  if (amax == 0.f) return 0;
  if ((b >> 23) == 0) return -126;  // below 2^-126: the clamp
  const int k = (int)(b >> 23) - 127 - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return k < -126 ? -126 : (k > 126 ? 126 : k);
}
__device__ __forceinline__ float pow2f(int k) { return __uint_as_float((uint32_t)(127 + k) << 23); }  // |k| <= 126

// Two E4M3 codes (round to nearest even, saturating): element lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_code(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Values of the two E4M3 codes in the low 16 bits of c (low byte -> lo),
// through the exact E4M3 -> f16 conversion and f16 -> f32.
__device__ __forceinline__ void e4m3x2_value(uint32_t c, float& lo, float& hi) {
  uint32_t h2;
  asm("{\n.reg .b16 t;\ncvt.u16.u32 t, %1;\ncvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(h2) : "r"(c));
  asm("{\n.reg .b16 a, b;\nmov.b32 {a, b}, %2;\ncvt.f32.f16 %0, a;\ncvt.f32.f16 %1, b;\n}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
}

// Clear the sign bit of every byte whose magnitude bits are zero (-0 -> 0).
__device__ __forceinline__ uint32_t drop_negative_zero_bytes(uint32_t w) {
  const uint32_t mag = w & 0x7F7F7F7Fu;
  const uint32_t nonzero = (mag + 0x7F7F7F7Fu) & 0x80808080u;
  return mag | (w & nonzero);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace nvfp4
