// Feature map of one dimension for the float32 decode steps (decode.cu, the
// fused stack step in stack.cu): fast hardware functions on reduced arguments.
#pragma once
#include "sanatan_math.cuh"

namespace sanatan {
namespace decm {

// sin and cos of x after reducing it into [-pi, pi] (the hardware sine and
// cosine are accurate to about 4e-7 there).
__device__ __forceinline__ void sincos_reduced(float x, float* s, float* c) {
  const float k = rintf(x * kInv2Pi);
  x = fmaf(-k, kC1, x);
  x = fmaf(-k, kC2, x);
  x = fmaf(-k, kC3, x);
  __sincosf(x, s, c);
}

// The six channels of one dimension for the decode step (eqs. (2)-(4)):
// theta = pi u / (1 + |u|); r = tanh(gamma (cos(theta + omega) - sin(theta +
// omega))) evaluated as 1 - 2 / (exp(2y) + 1); rotation by the reduced phase.
// Absolute error about 1e-6 per channel (the decode bar is 1e-5 on o).
__device__ __forceinline__ void feat_decode(float u, float gamma, float omega, float phase,
                                            float (&ch)[6]) {
  const float th = kPi * __fdividef(u, 1.0f + fabsf(u));
  float s1, c1;
  sincos_reduced(th + omega, &s1, &c1);
  const float e = __expf(2.0f * gamma * (c1 - s1));
  const float r = 1.0f - __fdividef(2.0f, e + 1.0f);
  float s2, c2;
  sincos_reduced(th + phase, &s2, &c2);
  ch[0] = 1.0f;
  ch[1] = c2;
  ch[2] = s2;
  ch[3] = r;
  ch[4] = r * c2;
  ch[5] = r * s2;
}

}  // namespace decm
}  // namespace sanatan
