// Device activations shared by every epilogue.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace fmlp {

// 2^v with the hardware's base-2 exponential (relative error about 2^-22; results below the
// normal range flush to zero).
__device__ __forceinline__ float ex2_approx(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// GELU, tanh form: 0.5 x (1 + tanh(z)), z = sqrt(2/pi) (x + 0.044715 x^3).
// Evaluated through the identity (1 + tanh z) / 2 = 1 / (1 + e^{-2z}) with
// e^{-2z} = 2^{x (c1 + c2 x^2)}, c1 = -2 sqrt(2/pi) log2(e) and c2 = 0.044715 c1 folded at
// compile time: one multiply, one multiply-add, one multiply, one base-2 exponential and one
// fast divide. As x -> -inf the exponential overflows to +inf and the quotient goes to 0 (the
// correct limit); as x -> +inf it returns x.
__device__ __forceinline__ float gelu_tanh_f(float x) {
  constexpr double kC1 = -2.0 * 0.79788456080286535588 * 1.44269504088896340736;
  const float c1 = static_cast<float>(kC1), c2 = static_cast<float>(kC1 * 0.044715);
  const float e = ex2_approx(x * fmaf(c2, x * x, c1));
  return __fdividef(x, 1.0f + e);
}

// GELU, exact form: 0.5 x (1 + erf(x / sqrt 2)), with erf from the rational approximation of
// Abramowitz and Stegun, Handbook of Mathematical Functions, eq. 7.1.26 (absolute error at
// most 1.5e-7): for z >= 0, erf z = 1 - q with q = (a1 t + a2 t^2 + ... + a5 t^5) e^{-z^2} and
// t = 1 / (1 + p z). Taking z = |x| / sqrt 2, erf being odd gives 1 + erf(x / sqrt 2) = 2 - q
// for x >= 0 and q for x < 0. One fast reciprocal, one base-2 exponential and six FMAs replace
// the library erff, which made the bias+GELU epilogue of a short-K GEMM three times slower
// than the MMAs it follows; the GELU error stays below 5e-7 absolute on [-12, 12].
__device__ __forceinline__ float gelu_erf_f(float x) {
  const float z = fabsf(x) * 0.70710678118654752f;
  const float t = __fdividef(1.0f, fmaf(0.3275911f, z, 1.0f));
  float poly = fmaf(1.061405429f, t, -1.453152027f);
  poly = fmaf(poly, t, 1.421413741f);
  poly = fmaf(poly, t, -0.284496736f);
  poly = fmaf(poly, t, 0.254829592f);
  // e^{-z^2} = 2^{-x^2 log2(e) / 2}
  const float q = poly * t * ex2_approx(x * x * static_cast<float>(-0.5 * 1.44269504088896340736));
  return 0.5f * x * (x >= 0.0f ? 2.0f - q : q);
}

// ---- two values at once (f32x2 arithmetic of sm_100 and later: one instruction, two lanes,
// each rounded to nearest like the scalar operation), for the GEMM epilogues, where the
// instruction count of the activation sets the pace of short-K tiles.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
  return v;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_splat(float v) { return f2_pack(v, v); }
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// 1/v with the hardware's approximate reciprocal (relative error about 2^-23).
__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// gelu_tanh on two values: the formula of gelu_tanh_f with x / (1 + e) taken as
// x * (1 / (1 + e)).
__device__ __forceinline__ uint64_t gelu_tanh_f2(uint64_t x) {
  constexpr double kC1 = -2.0 * 0.79788456080286535588 * 1.44269504088896340736;
  const uint64_t arg =
      f2_mul(x, f2_fma(f2_mul(x, x), f2_splat(static_cast<float>(kC1 * 0.044715)),
                       f2_splat(static_cast<float>(kC1))));
  float a0, a1;
  f2_unpack(arg, a0, a1);
  const uint64_t d = f2_add(f2_pack(ex2_approx(a0), ex2_approx(a1)), f2_splat(1.0f));
  float d0, d1;
  f2_unpack(d, d0, d1);
  return f2_mul(x, f2_pack(rcp_approx(d0), rcp_approx(d1)));
}

// gelu_erf on two values: the formula of gelu_erf_f (Abramowitz and Stegun 7.1.26).
__device__ __forceinline__ uint64_t gelu_erf_f2(uint64_t x) {
  float x0, x1;
  f2_unpack(x, x0, x1);
  const uint64_t d = f2_fma(f2_pack(fabsf(x0), fabsf(x1)),
                            f2_splat(static_cast<float>(0.3275911 * 0.70710678118654752)),
                            f2_splat(1.0f));
  float d0, d1;
  f2_unpack(d, d0, d1);
  const uint64_t t = f2_pack(rcp_approx(d0), rcp_approx(d1));
  uint64_t poly = f2_fma(f2_splat(1.061405429f), t, f2_splat(-1.453152027f));
  poly = f2_fma(poly, t, f2_splat(1.421413741f));
  poly = f2_fma(poly, t, f2_splat(-0.284496736f));
  poly = f2_fma(poly, t, f2_splat(0.254829592f));
  const uint64_t arg =
      f2_mul(f2_mul(x, x), f2_splat(static_cast<float>(-0.5 * 1.44269504088896340736)));
  float a0, a1;
  f2_unpack(arg, a0, a1);
  const uint64_t q = f2_mul(f2_mul(poly, t), f2_pack(ex2_approx(a0), ex2_approx(a1)));
  const uint64_t two_minus_q = f2_fma(q, f2_splat(-1.0f), f2_splat(2.0f));
  float q0, q1, w0, w1;
  f2_unpack(q, q0, q1);
  f2_unpack(two_minus_q, w0, w1);
  return f2_mul(f2_mul(x, f2_splat(0.5f)), f2_pack(x0 >= 0.0f ? w0 : q0, x1 >= 0.0f ? w1 : q1));
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
