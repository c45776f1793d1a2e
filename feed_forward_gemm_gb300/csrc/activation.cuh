// Device activations shared by every epilogue.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace fmlp {

// GELU, tanh form: 0.5 x (1 + tanh(z)), z = sqrt(2/pi) (x + 0.044715 x^3).
// Evaluated through the identity (1 + tanh z) / 2 = 1 / (1 + e^{-2z}), so one fast exponential
// and one fast divide replace tanh. As x -> -inf the exponential overflows to +inf and the
// quotient goes to 0 (the correct limit); as x -> +inf it returns x.
__device__ __forceinline__ float gelu_tanh_f(float x) {
  const float two_k = 1.5957691216057308f;          // 2 * sqrt(2 / pi)
  const float z2 = two_k * x * fmaf(0.044715f * x, x, 1.0f);
  return __fdividef(x, 1.0f + __expf(-z2));
}

// GELU, exact form: 0.5 x (1 + erf(x / sqrt 2)), with erf from the rational approximation of
// Abramowitz and Stegun, Handbook of Mathematical Functions, eq. 7.1.26 (absolute error at
// most 1.5e-7): for z >= 0, erf z = 1 - q with q = (a1 t + a2 t^2 + ... + a5 t^5) e^{-z^2} and
// t = 1 / (1 + p z). Taking z = |x| / sqrt 2, erf being odd gives 1 + erf(x / sqrt 2) = 2 - q
// for x >= 0 and q for x < 0. One fast reciprocal, one fast exponential and six FMAs replace
// the library erff, which made the bias+GELU epilogue of a short-K GEMM three times slower
// than the MMAs it follows; the GELU error stays below 5e-7 absolute on [-12, 12].
__device__ __forceinline__ float gelu_erf_f(float x) {
  const float z = fabsf(x) * 0.70710678118654752f;
  const float t = __fdividef(1.0f, fmaf(0.3275911f, z, 1.0f));
  float poly = fmaf(1.061405429f, t, -1.453152027f);
  poly = fmaf(poly, t, 1.421413741f);
  poly = fmaf(poly, t, -0.284496736f);
  poly = fmaf(poly, t, 0.254829592f);
  const float q = poly * t * __expf(-z * z);
  return 0.5f * x * (x >= 0.0f ? 2.0f - q : q);
}

// ReLU: max(x, 0), NaN passed through, -0 giving +0 (as torch's relu).
__device__ __forceinline__ float relu_f(float x) { return x > 0.0f ? x : (x != x ? x : 0.0f); }

// The hidden activation by mode: 0 GELU tanh, 1 GELU erf, 2 ReLU.
__device__ __forceinline__ float gelu_f(float x, int mode) {
  return mode == 2 ? relu_f(x) : (mode == 1 ? gelu_erf_f(x) : gelu_tanh_f(x));
}

// Two floats -> packed bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace fmlp
