// 2^x on the FMA pipe, for part of the softmax exponents.
//
// The special-function unit evaluates ex2 at a quarter of the FMA pipe's lane rate, and a
// softmax warpgroup spends most of its critical path there; computing a fixed share of
// the exponents with ordinary arithmetic moves that share to pipes that have room.
// Method (Cody and Waite's range reduction with a polynomial): x = j + f with
// j = round(x) and f = x - j in [-1/2, 1/2]; 2^f ~ p(f) by Horner's rule; 2^j by adding
// j to the exponent field of p(f).  Adding 1.5 * 2^23 to x rounds it to an integer held
// in the low mantissa bits, and shifting those bits left by 23 gives j's exponent-field
// increment in two's complement, so one integer multiply-add inserts it.  x is first
// clamped to >= -125, so 2^j p(f) stays a normal float (>= 2^-125 * 0.7); callers use
// this only where no exponent is masked to -inf (where a true 0 is needed).
// Coefficients: gen_exp2_poly.py (iterated weighted least squares towards the minimax
// relative error on [-1/2, 1/2]); worst relative error with float32 evaluation:
// degree 3: 7.5e-5, degree 4: 2.7e-6.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace zl {

template <int kDegree>
struct Exp2Poly;
template <>
struct Exp2Poly<3> {
  static constexpr float c[4] = {0x1.fff692p-1f, 0x1.62f31ap-1f, 0x1.f0de1ap-3f, 0x1.c3f76p-5f};
};
template <>
struct Exp2Poly<4> {
  static constexpr float c[5] = {0x1.ffffe8p-1f, 0x1.62e0dcp-1f, 0x1.ec06dap-3f, 0x1.ca1442p-5f, 0x1.3997d6p-7f};
};

// 2^x for a pair of arguments, two-wide arithmetic where it exists.
template <int kDegree>
__device__ __forceinline__ float2 exp2_poly2(float2 x) {
  constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
  x.x = fmaxf(x.x, -125.0f);
  x.y = fmaxf(x.y, -125.0f);
  const float2 t = __fadd2_rn(x, make_float2(kRound, kRound));
  const float2 j = __fadd2_rn(t, make_float2(-kRound, -kRound));
  const float2 f = __fadd2_rn(x, make_float2(-j.x, -j.y));
  // local constant copy (reading the static member in a constant expression keeps it
  // out of device memory)
  constexpr float c[] = {Exp2Poly<kDegree>::c[0], Exp2Poly<kDegree>::c[1], Exp2Poly<kDegree>::c[2],
                         Exp2Poly<kDegree>::c[3], Exp2Poly<kDegree>::c[kDegree >= 4 ? 4 : 3]};
  float2 p = make_float2(c[kDegree], c[kDegree]);
#pragma unroll
  for (int k = kDegree - 1; k >= 0; --k) p = __ffma2_rn(p, f, make_float2(c[k], c[k]));
  const uint32_t ex = __float_as_uint(t.x), ey = __float_as_uint(t.y);
  return make_float2(__uint_as_float(ex * (1u << 23) + __float_as_uint(p.x)),
                     __uint_as_float(ey * (1u << 23) + __float_as_uint(p.y)));
}

}  // namespace zl
