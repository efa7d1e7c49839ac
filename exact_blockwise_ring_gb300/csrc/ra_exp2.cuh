// ra_exp2.cuh -- 2^x in software on the FMA pipe, for a share of a softmax's
// exponentials beside the hardware exponential unit (MUFU ex2), which the softmax keeps
// busy.
//
// Method: Cody and Waite's range reduction, x = n + f with n = round(x) and f in
// [-1/2, 1/2], 2^x = 2^n p(f), where p(f) = 1 + f (c1 + f (c2 + f (c3 + f c4))) is the
// polynomial of that form (p(0) = 1, so an integer x gives exactly 2^n) with the smallest
// largest relative error over [-1/2, 1/2], found by the Remez exchange algorithm
// (exp2_poly.py prints the coefficients below, rounded to float32; relative error 3.6e-6).
// n comes from adding 1.5 * 2^23, after which the sum's low mantissa bits hold round(x);
// 2^n is built in the exponent field of a float.
//   x <= -127, including -inf, gives +0 (as the hardware unit's flush-to-zero form gives
//   for results below the normal range); NaN gives NaN; x must stay below 128.
#pragma once

#include <cstdint>

#include "ra_ptx.cuh"

namespace ra {

constexpr float kExp2C1 = 6.931136250e-01f;
constexpr float kExp2C2 = 2.402071059e-01f;
constexpr float kExp2C3 = 5.597688258e-02f;
constexpr float kExp2C4 = 9.782912210e-03f;

__device__ __forceinline__ float max_keep_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// 2^x0, 2^x1 for a packed pair.
__device__ __forceinline__ uint64_t exp2_soft_x2(float x0, float x1) {
  const uint64_t x = f2_pack(max_keep_nan(x0, -127.f), max_keep_nan(x1, -127.f));
  const uint64_t big = f2_pack(12582912.f, 12582912.f);          // 1.5 * 2^23
  const uint64_t t = f2_add(x, big);                              // low bits: round(x)
  const uint64_t f = f2_sub(x, f2_sub(t, big));                   // exact, in [-1/2, 1/2]
  uint64_t q = f2_fma(f2_pack(kExp2C4, kExp2C4), f, f2_pack(kExp2C3, kExp2C3));
  q = f2_fma(q, f, f2_pack(kExp2C2, kExp2C2));
  q = f2_fma(q, f, f2_pack(kExp2C1, kExp2C1));
  q = f2_fma(q, f, f2_pack(1.f, 1.f));
  // 2^n: the low nine bits of t's pattern are n mod 512, so (bits << 23) + (127 << 23)
  // is the pattern of 2^n for -127 < n < 128, and +0 for n = -127
  float t0, t1;
  f2_unpack(t, t0, t1);
  const float s0 = __uint_as_float((__float_as_uint(t0) << 23) + 0x3f800000u);
  const float s1 = __uint_as_float((__float_as_uint(t1) << 23) + 0x3f800000u);
  return f2_mul(q, f2_pack(s0, s1));
}

}  // namespace ra
