// 2^x on the FMA pipe, for softmax exponentials that would otherwise all queue
// on the SM's special-function unit (16 results per clock per SM, the same
// order as the tensor-core rate of an attention tile).
//
// Method: range reduction x = n + f with n = round(x) and f in [-1/2, 1/2]
// (the rounding is done by adding 1.5 * 2^23, which leaves n in the low
// mantissa bits), a degree-4 polynomial for 2^f, and the scaling by 2^n as an
// integer add into the exponent field.  The coefficients are a weighted
// least-squares fit of 2^f over Chebyshev nodes on [-1/2, 1/2], iterated toward
// the minimax relative error; evaluated in FP32 the relative error stays below
// 3e-6, far under the FP16 / BF16 rounding of the probabilities that follows.
// Inputs below -125 return 2^-125 (zero after FP16 rounding, negligible next to
// a softmax row sum of at least 1).
#pragma once

namespace qwen {

constexpr float kExp2C0 = 0.9999992847442627f;
constexpr float kExp2C1 = 0.6931217908859253f;
constexpr float kExp2C2 = 0.240247443318367f;
constexpr float kExp2C3 = 0.05591785907745361f;
constexpr float kExp2C4 = 0.009570101276040077f;

__device__ __forceinline__ float exp2_fma(float x) {
  x = fmaxf(x, -125.0f);
  const float t = x + 12582912.0f;  // 1.5 * 2^23
  const float n = t - 12582912.0f;
  const float f = x - n;
  float p = fmaf(kExp2C4, f, kExp2C3);
  p = fmaf(p, f, kExp2C2);
  p = fmaf(p, f, kExp2C1);
  p = fmaf(p, f, kExp2C0);
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

}  // namespace qwen
