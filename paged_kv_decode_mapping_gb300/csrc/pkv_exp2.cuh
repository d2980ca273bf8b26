// pkv_exp2.cuh -- 2^x on the FMA pipe, for the prefill softmax, whose special-function
// unit (the hardware ex2) would otherwise bound it: part of each row's exponentials go
// through this form instead, so both units work at once.
//
// Method: additive range reduction to the nearest integer, x = j + f with |f| <= 1/2
// (exact in binary floating point, so no split constant is needed), then a cubic
// polynomial for 2^f on [-1/2, 1/2] whose coefficients are the minimax fit for relative
// error found by the Remez exchange algorithm (max relative error 7.5e-5, about 2^-13.7,
// far inside the 2^-9 of the bf16 weights it feeds), then 2^j applied by adding j to the
// exponent field.
#pragma once

#include <stdint.h>

namespace pkv {
namespace dev {

// Remez minimax coefficients of 2^f ~ c0 + c1 f + c2 f^2 + c3 f^3 on [-1/2, 1/2].
constexpr float kExp2C0 = 0x1.fff692p-1f;
constexpr float kExp2C1 = 0x1.62f31ap-1f;
constexpr float kExp2C2 = 0x1.f0de1ap-3f;
constexpr float kExp2C3 = 0x1.c3f76p-5f;

// 2^x for x < 127.  Inputs below -125 are taken as -125, so the result stays a normal
// float (2^-125 weighs nothing against a row maximum near 1); NaN is taken as -125 too.
__device__ __forceinline__ float exp2_fma(float x) {
  constexpr float kRound = 12582912.f;  // 1.5 * 2^23: x + kRound holds rint(x) in its low bits
  x = fmaxf(x, -125.f);
  const float t = __fadd_rn(x, kRound);
  const int j = __float_as_int(t) - 0x4B400000;  // rint(x)
  const float f = __fsub_rn(x, __fsub_rn(t, kRound));  // x - j, in [-1/2, 1/2]
  const float p = fmaf(fmaf(fmaf(kExp2C3, f, kExp2C2), f, kExp2C1), f, kExp2C0);
  return __int_as_float(__float_as_int(p) + (int)((uint32_t)j << 23));
}

}  // namespace dev
}  // namespace pkv
