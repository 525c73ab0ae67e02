// angle.cuh -- the angle of the position phase rotation of queries and keys
// ("2. Relative Position via Complex Exponential Phase Rotations" of "RetNet
// Guide: Retentive Networks & The Impossible Triangle"): the pair (2j, 2j+1)
// of the query or key of the token at position p is turned by p theta_j.
#pragma once

#include <cuda_bf16.h>
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

// One bf16 pair (x, y) turned by the angle with cosine c and sine s, rounded
// to bf16 (round to nearest even).
__device__ __forceinline__ uint32_t rot_pair(uint32_t w, float c, float s) {
  const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  const __nv_bfloat162 o = __floats2bfloat162_rn(v.x * c - v.y * s, v.x * s + v.y * c);
  return *reinterpret_cast<const uint32_t*>(&o);
}

}  // namespace ret
