// Software 2^x on the FMA/ALU pipes: exact range reduction in base 2 followed by
// a cubic for 2^f (the exponential emulation of the FlashAttention-4 pages:
// "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
// Hardware Scaling", Summary — polynomial approximation after Cody-Waite range
// reduction, evaluated on the FMA units to relieve the MUFU unit).
//
// The input is already in base-2 units (the softmax folds scale*log2(e) into
// one FMA), so the reduction x = n + f, n = round(x), f in [-1/2, 1/2] is exact
// and no split constant is needed. n is obtained by adding 1.5*2^23, which
// leaves round(x) in the low mantissa bits; 2^n is applied by adding n to the
// exponent field of q(f). Relative error <= 2^-13 for x in [-125, 8]; inputs
// below -127 (including -inf) return +0; between -127 and -125 the result is
// below 2^-125 in magnitude.
#pragma once
#include <cstdint>
#include <cstring>

#include "exp2_poly_coeffs.h"

namespace fa {

__host__ __device__ __forceinline__ float exp2_poly(float x) {
#ifdef __CUDA_ARCH__
  x = fmaxf(x, -127.0f);
  const float t = __fadd_rn(x, 12582912.0f);
  const float n = __fsub_rn(t, 12582912.0f);
  const float f = __fsub_rn(x, n);
  const float q = __fmaf_rn(__fmaf_rn(__fmaf_rn(FA_EXP2_C3, f, FA_EXP2_C2), f, FA_EXP2_C1), f, 1.0f);
  const int bits = __float_as_int(q) + (__float_as_int(t) << 23);
  return __int_as_float(bits);
#else
  // Host twin of the device sequence (same operations, each correctly rounded).
  x = x > -127.0f ? x : -127.0f;
  volatile float t = x + 12582912.0f;
  volatile float n = t - 12582912.0f;
  volatile float f = x - n;
  const float q = fmaf(fmaf(fmaf(FA_EXP2_C3, f, FA_EXP2_C2), f, FA_EXP2_C1), f, 1.0f);
  uint32_t qb, tb;
  float tt = t;
  memcpy(&qb, &q, 4);
  memcpy(&tb, &tt, 4);
  const uint32_t rb = qb + (tb << 23);
  float r;
  memcpy(&r, &rb, 4);
  return r;
#endif
}

}  // namespace fa
