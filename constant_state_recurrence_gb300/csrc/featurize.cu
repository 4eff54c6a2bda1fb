// Elementwise feature map Phi (reading notes §2.2-§2.3, paper eqs. (2)-(6)).
#include "sanatan_internal.h"
#include "sanatan_math.cuh"

namespace sanatan {
namespace {

// One thread per (b, h, t, a) element writes the six channels of dimension a.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) featurize_kernel(const Tin* __restrict__ u,
                                                        const float* __restrict__ gamma,
                                                        const float* __restrict__ omega,
                                                        const float* __restrict__ phi,
                                                        Tout* __restrict__ out, int H, int T,
                                                        int d, int64_t pos0, int64_t total) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int a = static_cast<int>(idx % d);
  const int64_t row = idx / d;  // (b*H + h)*T + i
  const int i = static_cast<int>(row % T);
  const int h = static_cast<int>((row / T) % H);
  const float ph = phase_mod_2pi(pos0 + i, phi[h * d + a]);
  const FeatAngles f = feat_exact(load_as_float(u + idx), gamma[h], omega[h * d + a], ph);
  float ch[6];
  feat_channels(f, ch);
  Tout* dst = out + idx * 6;
#pragma unroll
  for (int c = 0; c < 6; ++c) dst[c] = store_from_float<Tout>(ch[c]);
}

template <typename Tin, typename Tout>
cudaError_t launch(const void* u, const float* gamma, const float* omega, const float* phi,
                   void* out, int B, int H, int T, int d, int64_t pos0, cudaStream_t st) {
  const int64_t total = static_cast<int64_t>(B) * H * T * d;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  featurize_kernel<Tin, Tout><<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      static_cast<const Tin*>(u), gamma, omega, phi, static_cast<Tout*>(out), H, T, d, pos0,
      total);
  return cudaGetLastError();
}

// The rotation rate from its unconstrained parameter (reading notes §2.2,
// eq. (4)): phi = scale tanh(lambda_raw), and the pull-back of a rate
// gradient, dlambda_raw = dphi scale (1 - tanh^2(lambda_raw)).
__global__ void __launch_bounds__(256) rate_kernel(const float* __restrict__ raw,
                                                   const float* __restrict__ dphi, int n,
                                                   float scale, float* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float t = tanhf(raw[i]);
  out[i] = dphi == nullptr ? scale * t : dphi[i] * scale * (1.0f - t * t);
}

}  // namespace

cudaError_t rate_launch(const float* raw, const float* dphi, int n, float scale, float* out,
                        cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  rate_kernel<<<(n + 255) / 256, 256, 0, st>>>(raw, dphi, n, scale, out);
  return cudaGetLastError();
}

cudaError_t featurize_launch(const void* u, int u_dtype, const float* gamma,
                             const float* omega, const float* phi, int B, int H, int T, int d,
                             int64_t pos0, void* out, int out_dtype, cudaStream_t st) {
  if (u_dtype == SANATAN_F32 && out_dtype == SANATAN_F32)
    return launch<float, float>(u, gamma, omega, phi, out, B, H, T, d, pos0, st);
  if (u_dtype == SANATAN_F32 && out_dtype == SANATAN_BF16)
    return launch<float, __nv_bfloat16>(u, gamma, omega, phi, out, B, H, T, d, pos0, st);
  if (u_dtype == SANATAN_BF16 && out_dtype == SANATAN_F32)
    return launch<__nv_bfloat16, float>(u, gamma, omega, phi, out, B, H, T, d, pos0, st);
  return launch<__nv_bfloat16, __nv_bfloat16>(u, gamma, omega, phi, out, B, H, T, d, pos0, st);
}

}  // namespace sanatan
