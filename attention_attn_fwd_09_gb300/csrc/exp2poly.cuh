// Software 2^x on the FMA pipe: range reduction x = floor(x) + f, 2^floor(x) put into the
// exponent field with integer arithmetic, 2^f from a cubic.
//
// Follows "Hotelren FA4 summary", section 3.2 (polynomial exponential: split x into its
// integer and fractional parts, integer part by bit manipulation, cubic for the fraction)
// and "FlashAttention-4 explained", section 04, trick one (e^x ~ 2^n (p0 + p1 f + p2 f^2 +
// p3 f^3), computed by the otherwise idle FMA units).  The coefficients are this
// library's own minimax fit (fit_exp2.py -> exp2_coeffs.h), constrained to p(0) = 1.
#pragma once
#include "exp2_coeffs.h"

namespace attn {

// floor(x) without a conversion instruction: adding 1.5 * 2^23 with round-toward-minus-
// infinity leaves floor(x) in the low mantissa bits of t (|x| < 2^22).  Because the low
// nine bits of the bit pattern of 1.5 * 2^23 are zero, (bits(t) << 23) == floor(x) << 23.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23

// Production form.  Inputs below -127 (including -inf from masking) clamp to -127, which
// gives exactly +0 because p(0) == 1.  Results for x in (-127, -126) are not the correct
// subnormals (they are below 2^-126 either way and cannot change a bf16 probability).
__device__ __forceinline__ float exp2_poly(float x) {
  x = fmaxf(x, -127.0f);
  const float t = __fadd_rd(x, kRoundMagic);
  const float f = x - (t - kRoundMagic);  // exact, in [0, 1)
  const float p = fmaf(fmaf(fmaf(ATTN_EXP2_C3, f, ATTN_EXP2_C2), f, ATTN_EXP2_C1), f, ATTN_EXP2_C0);
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

// Same polynomial, correct over the whole of [-127, 0] including the fp32 subnormal
// range: for floor(x) = -127 it scales by 2^-126 and then halves with a rounded
// multiply (compile without flush-to-zero).  Used by the accuracy test entry point.
__device__ __forceinline__ float exp2_poly_full_range(float x) {
  x = fmaxf(x, -127.0f);
  const float t = __fadd_rd(x, kRoundMagic);
  const float n = t - kRoundMagic;
  const float f = x - n;
  const float p = fmaf(fmaf(fmaf(ATTN_EXP2_C3, f, ATTN_EXP2_C2), f, ATTN_EXP2_C1), f, ATTN_EXP2_C0);
  if (n >= -126.0f) return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
  const float hi = __int_as_float(__float_as_int(p) + ((__float_as_int(t) + 1) << 23));
  return __fmul_rn(hi, 0.5f);
}

}  // namespace attn
