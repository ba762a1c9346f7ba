// 2^x on the FMA pipe, for a pair of fp32 values at once (f32x2 instructions).
//
// Cody-Waite range reduction: n = round(x) (adding and subtracting 1.5 * 2^23
// rounds to the nearest integer under round-to-nearest), f = x - n in
// [-1/2, 1/2] exactly, 2^f by a cubic, and 2^n applied by adding n to the
// exponent field.  Inputs are clamped below at -126 so the exponent stays in
// range; below that the result is at most 2^-126 (about 1e-38) instead of the
// exact tiny value.  Relative error about 7.5e-5 (see exp2_poly.py).
#pragma once

#include "ptx.cuh"

namespace attn_sink {

// Cubic minimax fit of 2^f on [-1/2, 1/2] for relative error, printed by
// exp2_poly.py (Lawson's iteratively reweighted least squares).
constexpr float kExp2C0 = 9.999280572e-01f;
constexpr float kExp2C1 = 6.932610273e-01f;
constexpr float kExp2C2 = 2.426112145e-01f;
constexpr float kExp2C3 = 5.517137796e-02f;
constexpr float kRoundMagic = 12582912.f;  // 1.5 * 2^23

__device__ __forceinline__ void exp2_poly_pair(float x0, float x1, float& y0, float& y1) {
  const uint64_t x = f2_pack(fmaxf(x0, -126.f), fmaxf(x1, -126.f));
  const uint64_t t = f2_add(x, f2_pack(kRoundMagic, kRoundMagic));      // magic + n
  const uint64_t r = f2_add(t, f2_pack(-kRoundMagic, -kRoundMagic));    // n
  const uint64_t f = f2_fma(r, f2_pack(-1.f, -1.f), x);                 // x - n
  uint64_t p = f2_fma(f2_pack(kExp2C3, kExp2C3), f, f2_pack(kExp2C2, kExp2C2));
  p = f2_fma(p, f, f2_pack(kExp2C1, kExp2C1));
  p = f2_fma(p, f, f2_pack(kExp2C0, kExp2C0));
  float p0, p1, t0, t1;
  f2_unpack(p, p0, p1);
  f2_unpack(t, t0, t1);
  // The low bits of magic + n hold n (two's complement); shifting by 23 drops
  // the magic's own bits and lands n in the exponent field.
  y0 = __uint_as_float(__float_as_uint(p0) + (__float_as_uint(t0) << 23));
  y1 = __uint_as_float(__float_as_uint(p1) + (__float_as_uint(t1) << 23));
}

}  // namespace attn_sink
