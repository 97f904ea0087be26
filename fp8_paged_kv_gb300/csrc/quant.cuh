// quant.cuh -- the division at the heart of the e4m3 quantiser, x / scale,
// for a scale shared by a whole tensor.
#pragma once

#include "common.cuh"

namespace fpk {

// Quotient x / s for a divisor used many times (the per-tensor quantiser
// scale), by Markstein's division (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Develop. 34,
// 1990): with r = RN(1/s), q0 = RN(x r) is within one ulp of x / s; the
// residual x - q0 s is exact as one FMA, and RN(q0 + residual r) is the
// correctly rounded quotient whenever it lies in the normal range.  Below
// that (|x / s| < 2^-126) the result may differ from RN(x / s) by an ulp of a
// subnormal -- far below 2^-10, where every such value encodes to a zero e4m3
// code of the same sign.  Zero, infinite and NaN q0 are returned unchanged;
// a divisor whose reciprocal is not a normal number takes the IEEE division.
struct Divisor {
  float s, r;
  bool recip_ok;
};
__device__ __forceinline__ Divisor make_divisor(float s) {
  Divisor d;
  d.s = s;
  d.r = __frcp_rn(s);
  d.recip_ok = isfinite(d.r) && fabsf(d.r) >= 1.17549435e-38f;
  return d;
}
// The corrected product alone, for a divisor with d.recip_ok.  A zero,
// infinite or NaN q0 is the answer as it is (this keeps the sign of -0 and
// the infinity of an overflowing quotient).
__device__ __forceinline__ float div_fast(float x, const Divisor& d) {
  const float q0 = __fmul_rn(x, d.r);
  const float e = __fmaf_rn(-q0, d.s, x);
  const float q = __fmaf_rn(e, d.r, q0);
  return (q0 != 0.f && fabsf(q0) <= 3.40282347e38f) ? q : q0;
}
__device__ __forceinline__ float div_by(float x, const Divisor& d) {
  return d.recip_ok ? div_fast(x, d) : __fdiv_rn(x, d.s);
}

}  // namespace fpk
