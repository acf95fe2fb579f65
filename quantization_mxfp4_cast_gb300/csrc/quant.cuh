// Block quantizer shared by the cast kernels and the GEMM epilogue that
// casts its own output: E2M1 (and the E8M0 block scale) of one 32-element
// block of fp32 values, NaN-propagating block amax, and the 32-point
// Hadamard normalization constant.
//
// Method: jax-aiter README, "Supported ops" table, row "MXFP4 Cast" (E2M1
// elements with E8M0 block scales).  Readings: scale byte
// max(floor(log2 amax) - 2 + 127, 0), NaN/Inf block -> 0xFF with codes 0,
// round to nearest even with saturation at 6, sign kept.
#pragma once

#include <stdint.h>

namespace mxfp4 {

// E2M1 codes of 8 values, element 0 in the low nibble of byte 0.  The
// conversion rounds to nearest even and saturates at +-6.
__device__ __forceinline__ uint32_t cvt8_e2m1(float v0, float v1, float v2, float v3, float v4,
                                              float v5, float v6, float v7) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return out;
}

// From the largest magnitude's bit pattern: scale byte and the exact
// power-of-two multiplier 2^-e (as fp32, and as a bf16 bit pattern).  For a
// finite amax with biased exponent E, floor(log2 amax) - kEmax + 127 =
// E - kEmax, clamped at 0 (E = 0 covers zero and subnormals); kEmax is the
// exponent of the element format's largest value (E2M1: 6 = 1.5 * 2^2 -> 2;
// E4M3: 448 = 1.75 * 2^8 -> 8).
struct BlockScale {
  uint32_t byte;
  float mult;
  uint32_t mult_bf16;
  bool nonfinite;
};

template <int kEmax = 2>
__device__ __forceinline__ BlockScale block_scale(uint32_t amax_bits) {
  BlockScale s;
  s.nonfinite = amax_bits >= 0x7F800000u;
  const int e_biased = static_cast<int>(amax_bits >> 23);
  const int byte = e_biased > kEmax ? e_biased - kEmax : 0;
  s.mult = __uint_as_float(static_cast<uint32_t>(254 - byte) << 23);
  s.mult_bf16 = static_cast<uint32_t>(254 - byte) << 7;
  s.byte = s.nonfinite ? 0xFFu : static_cast<uint32_t>(byte);
  return s;
}

// Codes of 8 fp32 elements under the block's scale (the conversion keeps the
// sign of values that round to zero, so no fix-up is needed).
__device__ __forceinline__ uint32_t quantize8(const float* y, const BlockScale& s) {
  if (s.nonfinite) return 0u;
  const float m = s.mult;
  return cvt8_e2m1(__fmul_rn(y[0], m), __fmul_rn(y[1], m), __fmul_rn(y[2], m),
                   __fmul_rn(y[3], m), __fmul_rn(y[4], m), __fmul_rn(y[5], m),
                   __fmul_rn(y[6], m), __fmul_rn(y[7], m));
}

// fp32 value nearest to 1/sqrt(32).
constexpr float kInvSqrt32 = 0x1.6a09e6p-3f;  // bit pattern 0x3E3504F3

// max(|a|, |b|, |c|) with NaN propagation (three-input form).
__device__ __forceinline__ float max3_nan_abs(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(fabsf(a)), "f"(fabsf(b)), "f"(fabsf(c)));
  return r;
}

// NaN-propagating max |v| of 32 fp32 values read as v(i), i = 0..31, in four
// independent chains of three-input maxima.
template <typename F>
__device__ __forceinline__ float amax32(F v) {
  float c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int b = 8 * k;
    float m = max3_nan_abs(v(b), v(b + 1), v(b + 2));
    m = max3_nan_abs(m, v(b + 3), v(b + 4));
    m = max3_nan_abs(m, v(b + 5), v(b + 6));
    c[k] = max3_nan_abs(m, v(b + 7), 0.f);
  }
  return max3_nan_abs(c[0], c[1], max3_nan_abs(c[2], c[3], 0.f));
}

// Elementwise max(|a|, |b|) of bf16 pairs, NaN-propagating (sign bits of
// the result are the XOR of the inputs' and must be masked off).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Packed fp32 pairs (Blackwell f32x2 arithmetic, IEEE round-to-nearest per lane).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float lo2(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi2(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// fp32 value of the bf16 element in the low (kHi = false) or high half of w,
// times s (a bf16 bit pattern), by the mixed-precision fma with -0 added:
// for a power-of-two s the product is exact in fp32 down to 2^-126 (anything
// smaller has |v| < 1/4 and gives a signed zero code either way), and adding
// -0 keeps the sign of a zero product.  With s = 1 this is the plain widening.
template <bool kHi>
__device__ __forceinline__ float bf16_times(uint32_t w, uint16_t s) {
  float r;
  if constexpr (kHi)
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tfma.rn.f32.bf16 %0, h, %2, 0f80000000;\n\t}"
        : "=f"(r) : "r"(w), "h"(s));
  else
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tfma.rn.f32.bf16 %0, l, %2, 0f80000000;\n\t}"
        : "=f"(r) : "r"(w), "h"(s));
  return r;
}
constexpr uint16_t kBf16One = 0x3F80;

// Codes of the 8 bf16 elements in 4 packed words (element 2i in the low half
// of word i), scaled by the power of two s (bf16 bit pattern).
__device__ __forceinline__ uint32_t quantize8_bf16(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                                   uint16_t s) {
  return cvt8_e2m1(bf16_times<false>(w0, s), bf16_times<true>(w0, s), bf16_times<false>(w1, s),
                   bf16_times<true>(w1, s), bf16_times<false>(w2, s), bf16_times<true>(w2, s),
                   bf16_times<false>(w3, s), bf16_times<true>(w3, s));
}

// Packed bf16 magnitude max of 2^n words as a balanced tree (independent
// operations instead of one serial chain).  Sign bits of the result are
// meaningless.
template <int kN>
__device__ __forceinline__ uint32_t tree_absmax_bf16x2(const uint32_t* w) {
  uint32_t m[kN / 2];
#pragma unroll
  for (int i = 0; i < kN / 2; ++i) m[i] = absmax_bf16x2(w[2 * i], w[2 * i + 1]);
#pragma unroll
  for (int n = kN / 4; n >= 1; n >>= 1) {
#pragma unroll
    for (int i = 0; i < n; ++i) m[i] = absmax_bf16x2(m[2 * i], m[2 * i + 1]);
  }
  return m[0];
}

// One block of 32 bf16 values in 16 packed words (element 2i in the low half
// of word i), no transform: packed magnitude max for the scale, then each
// element widened and scaled by the mixed-precision fma.  codes[g] holds
// elements 8g .. 8g+7.
__device__ __forceinline__ BlockScale quantize_bf16_block(const uint32_t (&w)[16], uint32_t (&codes)[4]) {
  uint32_t m = tree_absmax_bf16x2<16>(w);
  m = absmax_bf16x2(m, __byte_perm(m, 0, 0x1032));  // both halves hold the block max
  const BlockScale s = block_scale((m & 0x7FFFu) << 16);
  const uint16_t mb = static_cast<uint16_t>(s.mult_bf16);
#pragma unroll
  for (int g = 0; g < 4; ++g)
    codes[g] = s.nonfinite ? 0u : quantize8_bf16(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3], mb);
  return s;
}

// One block of 32 fp32 values through the orthonormal 32-point Walsh-Hadamard
// transform, then quantized.  Butterflies over strides 1, 2, 4, 8, 16: stride
// 1 in scalar fp32, the others on f32x2 pairs of neighbouring elements
// (elements 2i + e and 2(i + h/2) + e meet in the same half of a pair), each
// half an IEEE round-to-nearest add or subtract, so the numbers are those of
// the scalar order.  The block amax of RN(y / sqrt(32)) is RN(max |y| *
// RN(1/sqrt(32))) (rounding is monotonic).  The element value RN(y * c) * 2^-e
// equals RN(y * (c * 2^-e)) while c * 2^-e stays normal (scale byte <= 250)
// and any RN(y * c) below 2^-126 codes to a signed zero either way (byte >= 3),
// so that range takes one multiply and the rest two.  y is overwritten.
__device__ __forceinline__ BlockScale quantize_hadamard_block(float (&y)[32], uint32_t (&codes)[4]) {
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float a = y[j], c = y[j + 1];
    y[j] = __fadd_rn(a, c);
    y[j + 1] = __fsub_rn(a, c);
  }
  uint64_t z[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) z[i] = pk2(y[2 * i], y[2 * i + 1]);
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & h) continue;
      const uint64_t a = z[i], c = z[i + h];
      z[i] = add2(a, c);
      z[i + h] = sub2(a, c);
    }
  }
  const float amax = amax32([&](int i) { return (i & 1) ? hi2(z[i >> 1]) : lo2(z[i >> 1]); });
  const BlockScale s = block_scale(__float_as_uint(__fmul_rn(amax, kInvSqrt32)));
  if (s.byte - 3u <= 247u) {
    const float cm = __fmul_rn(kInvSqrt32, s.mult);
    const uint64_t m2 = pk2(cm, cm);
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = mul2(z[i], m2);
  } else {
    const uint64_t c2 = pk2(kInvSqrt32, kInvSqrt32), m2 = pk2(s.mult, s.mult);
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = mul2(mul2(z[i], c2), m2);
  }
#pragma unroll
  for (int g = 0; g < 4; ++g)
    codes[g] = s.nonfinite ? 0u
                           : cvt8_e2m1(lo2(z[4 * g]), hi2(z[4 * g]), lo2(z[4 * g + 1]), hi2(z[4 * g + 1]),
                                       lo2(z[4 * g + 2]), hi2(z[4 * g + 2]), lo2(z[4 * g + 3]),
                                       hi2(z[4 * g + 3]));
  return s;
}

}  // namespace mxfp4
