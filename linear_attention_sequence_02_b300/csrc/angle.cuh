// angle.cuh -- the angle of the position phase rotation of queries and keys
// ("2. Relative Position via Complex Exponential Phase Rotations" of "RetNet
// Guide: Retentive Networks & The Impossible Triangle"): the pair (2j, 2j+1)
// of the query or key of the token at position p is turned by p theta_j.
#pragma once

#include <cstdint>

namespace ret {

// 2 pi = kTwoPiHi + kTwoPiLo + ~7e-15: kTwoPiHi is 2 pi rounded to float,
// kTwoPiLo the remainder rounded to float.
constexpr float kTwoPiHi = 0x1.921fb6p+2f;
constexpr float kTwoPiLo = -0x1.777a5cp-23f;
constexpr float kInvTwoPi = 0x1.45f306p-3f;

// The angle p theta reduced to about [-pi, pi] by the method of Cody and
// Waite: the product is first split exactly into two floats, so positions p
// up to 2^24 (integers, exact in float) keep ~1e-7 rad of accuracy.
__device__ __forceinline__ float reduced_angle(float p, float theta) {
  const float hi = p * theta;
  const float lo = fmaf(p, theta, -hi);  // p theta = hi + lo exactly
  const float k = rintf(hi * kInvTwoPi);
  float r = fmaf(-k, kTwoPiHi, hi);  // exact: the difference needs at most 24 bits
  r = fmaf(-k, kTwoPiLo, r);
  return r + lo;
}

// One bf16 pair (x in the low half, y in the high half) turned by the angle
// with cosine c and sine s, rounded to bf16 (round to nearest even).  A bf16
// is the upper half of the float with the same bits, so unpacking is a shift
// and a mask.
__device__ __forceinline__ uint32_t rot_pair(uint32_t w, float c, float s) {
  const float x = __uint_as_float(w << 16), y = __uint_as_float(w & 0xffff0000u);
  const float ox = fmaf(x, c, -y * s), oy = fmaf(x, s, y * c);
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(oy), "f"(ox));  // oy to the high half
  return r;
}

}  // namespace ret
