// Device math for the SANATAN feature map.
//
// Feature map of "SANATAN: Root-Parity Gated Angular Attention with an Exact
// Constant-State Recurrent Form" (reading notes §2.2-§2.3, paper eqs. (2)-(6)):
//   theta     = pi * u / (1 + |u|)                                  eq. (2)
//   r         = tanh(gamma * (cos(theta + omega) - sin(theta + omega)))  eq. (3)
//   theta_rot = theta + t * phi                                     eq. (4)
//   Phi_a     = [1, cos theta_rot, sin theta_rot, r, r cos, r sin]  eq. (6)
// The root r uses the angle before the rotation.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace sanatan {

constexpr float kPi = 3.14159265358979323846f;
constexpr float kInv2Pi = 0.15915493667125702f;
// 2*pi = kC1 + kC2 + kC3 with kC1, kC2 holding 11 significant bits each, so
// that k * kC1 and k * kC2 are exact in float32 for |k| < 2^13 (Cody and
// Waite's additive range reduction).
constexpr float kC1 = 6.28125f;
constexpr float kC2 = 0.0019350051879882812f;
constexpr float kC3 = 3.019916050561733e-07f;
constexpr double kTwoPiD = 6.283185307179586476925286766559;

// Float64 reduction for positions or rates outside the float fast range.
// Kept out of line: float64 is far slower than float32 on this GPU, and an
// inlined copy could be evaluated (if-converted) even when not taken.
static __device__ __noinline__ float phase_mod_2pi_f64(int64_t t, float phi) {
  const double p = static_cast<double>(t) * static_cast<double>(phi);
  const double k = rint(p * (1.0 / kTwoPiD));
  return static_cast<float>(fma(-k, kTwoPiD, p));
}

// t * phi reduced into [-pi, pi] to about 3e-7 rad.  The product is kept as an
// exact float pair (FMA two-product) and reduced by the three-part 2*pi above;
// positions or rates outside the float fast range take the float64 path.
__device__ __forceinline__ float phase_mod_2pi(int64_t t, float phi) {
  if (t > -(1LL << 24) && t < (1LL << 24)) {
    const float tf = static_cast<float>(t);
    const float p_hi = tf * phi;
    if (fabsf(p_hi) < 51000.0f) {
      const float p_lo = fmaf(tf, phi, -p_hi);
      const float k = rintf(p_hi * kInv2Pi);
      float r = fmaf(-k, kC1, p_hi);
      r = fmaf(-k, kC2, r);
      return r + fmaf(-k, kC3, p_lo);
    }
  }
  return phase_mod_2pi_f64(t, phi);
}

// theta = pi u / (1 + |u|), correctly rounded division.
__device__ __forceinline__ float squash_exact(float u) { return kPi * u / (1.0f + fabsf(u)); }

struct FeatAngles {
  float c;  // cos(theta_rot)
  float s;  // sin(theta_rot)
  float r;  // soft root from the un-rotated theta
};

// Accurate float32 evaluation (libm-quality sincos/tanh); `phase` is t*phi
// already reduced by phase_mod_2pi.
__device__ __forceinline__ FeatAngles feat_exact(float u, float gamma, float omega, float phase) {
  const float th = squash_exact(u);
  float sx, cx;
  sincosf(th + omega, &sx, &cx);
  FeatAngles f;
  f.r = tanhf(gamma * (cx - sx));
  sincosf(th + phase, &f.s, &f.c);
  return f;
}

// The six channels of one dimension, channel order [1, c, s, r, r c, r s].
__device__ __forceinline__ void feat_channels(const FeatAngles& f, float out[6]) {
  out[0] = 1.0f;
  out[1] = f.c;
  out[2] = f.s;
  out[3] = f.r;
  out[4] = f.r * f.c;
  out[5] = f.r * f.s;
}

template <typename T>
__device__ __forceinline__ float load_as_float(const T* p);
template <>
__device__ __forceinline__ float load_as_float<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_as_float<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ T store_from_float(float x);
template <>
__device__ __forceinline__ float store_from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 store_from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

}  // namespace sanatan
