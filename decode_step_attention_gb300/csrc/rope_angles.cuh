// RoPE angles shared by the rotation kernels: inv_freq_i in fp64 from the host
// (theta^(-2i/D), or a caller's table such as a context-extension one) and the same
// frequencies as 64-bit fractions of a turn, from which the angle phi = p * inv_freq_i
// is reduced exactly in integer arithmetic before sin and cos are taken in fp32 (at
// p ~ 1.3e5 an fp32 product would already be off by ~1e-2 rad; fp64 arithmetic runs at
// a small fraction of the fp32 rate on this GPU).
#pragma once

#include <math.h>

namespace decattn {

struct InvFreq {
  double v[64];  // i = 0 .. D/2 - 1
};

// 2*pi split into a double head and the double nearest the remainder.
constexpr double kTwoPiHi = 6.283185307179586;
constexpr double kTwoPiLo = 2.4492935982947064e-16;
constexpr double kInvTwoPi = 0.15915494309189535;

// A rotated K element again, in fp64, for the rare element whose fp32 result cancels:
// own and other are the exact pre-rotation values of this element and its pair partner
// (the raw bf16 value, or its product with a bf16 norm weight, which fp32 holds
// exactly), rstd the head's QK-norm scale (1 without it). The first element of a pair
// becomes own cos - other sin, the second own cos + other sin. The fp32 path's error is a
// few 2^-24 of |own| + |other|; when the result is smaller than about 2^-12 of that,
// the error would exceed half a bf16 ulp of the result, and this path keeps the stored
// bf16 within one ulp of the exact rotation. (fp64 runs at a small fraction of the fp32
// rate here, so only those elements take it.)
__device__ __noinline__ inline float rope_exact(int p, double inv_freq, float own, float other,
                                                float rstd, bool second) {
  const double phi = (double)p * inv_freq;
  const double k = rint(phi * kInvTwoPi);
  double r = fma(-k, kTwoPiHi, phi);
  r = fma(-k, kTwoPiLo, r);
  double s, c;
  sincos(r, &s, &c);
  const double o = second ? (double)other : -(double)other;
  return (float)(fma((double)own, c, o * s) * (double)rstd);
}

// Whether a fp32 rotation result y of a pair whose normalised values have magnitudes
// a and b cancels enough to be formed again by rope_exact.
__device__ __forceinline__ bool rope_cancels(float y, float a, float b) {
  return fabsf(y) < 0x1p-11f * (fabsf(a) + fabsf(b));
}

// Host: the plain table theta^(-2i/D) for head_dim D.
InvFreq make_inv_freq(int D, double theta);

// The angles without fp64 arithmetic on the device. turns_i = inv_freq_i / (2 pi) as a
// 64-bit binary fraction (units of 2^-64 of a turn), rounded on the host; then p * turns_i computed
// modulo 2^64 is the angle's fractional turn exactly (the whole turns fall off the top),
// and its top 32 bits, read as a signed integer, give radians in [-pi, pi) after the
// rounding to fp32 (the angle is within 2^-32 of a turn plus that rounding).
struct RopeTurns {
  unsigned long long v[64];
};
// Every inv_freq_i must lie in [0, 1], so that turns_i < 1/(2 pi) fits the fraction.
RopeTurns make_rope_turns(int D, const InvFreq &inv);

__device__ __forceinline__ void rope_sincos_turns(int p, unsigned long long turns, float &s,
                                                  float &c) {
  const unsigned long long t = (unsigned long long)(unsigned)p * turns;
  const int hi = (int)(t >> 32);
  const float r = (float)hi * 1.4629180792671596e-09f;  // 2 pi / 2^32
  sincosf(r, &s, &c);
}

}  // namespace decattn
