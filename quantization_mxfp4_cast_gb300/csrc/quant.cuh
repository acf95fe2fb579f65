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

// One 32-element block held in registers, quantized in the plain order of the
// definition: optional orthonormal Walsh-Hadamard transform (fp32 butterflies
// over strides 1, 2, 4, 8, 16, then a multiply by RN(1/sqrt(32))), block amax,
// scale, E2M1 codes.  y is transformed in place; codes[g] holds elements
// 8g .. 8g+7.
__device__ __forceinline__ BlockScale quantize_block32(float (&y)[32], bool hadamard, uint32_t (&codes)[4]) {
  if (hadamard) {
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j & h) continue;
        const float a = y[j], c = y[j + h];
        y[j] = __fadd_rn(a, c);
        y[j + h] = __fsub_rn(a, c);
      }
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) y[j] = __fmul_rn(y[j], kInvSqrt32);
  }
  const BlockScale s = block_scale(__float_as_uint(amax32([&](int i) { return y[i]; })));
#pragma unroll
  for (int g = 0; g < 4; ++g) codes[g] = quantize8(y + 8 * g, s);
  return s;
}

}  // namespace mxfp4
