// All-float32 chunked forward on the CUDA cores (the f32-operand path).
//
// Per (batch, head) one CTA walks the sequence in chunks of kC tokens.  Inside
// a chunk the causal scores are formed explicitly; everything before the chunk
// is carried by the state (S, z) of reading notes §2.7 (paper eq. (9)):
//   N_t = sum_{j in chunk, j<=t} s_tj v_j + Phi(q_t)^T S_prev
//   D_t = sum_{j in chunk, j<=t} s_tj     + Phi(q_t)^T z_prev
//   o_t = N_t / (D_t + eps),  then  S += Phi(K)^T V,  z += Phi(K)^T 1.
// This is the same sum as the recurrence, re-associated by chunks.
#include "sanatan_internal.h"
#include "sanatan_math.cuh"

namespace sanatan {
namespace {

constexpr int kD = 64;
constexpr int kDv = 64;
constexpr int kF = 6 * kD;
constexpr int kFP = kF + 1;  // padded feature stride (bank spread across rows)
constexpr int kC = 32;
constexpr int kThreads = 256;

struct SimtSmem {
  float pq[kC * kFP];
  float pk[kC * kFP];
  float v[kC * kDv];
  float S[kF * kDv];
  float z[kF];
  float P[kC * (kC + 1)];
};

template <typename Tin>
__global__ void __launch_bounds__(kThreads, 1) chunk_fwd_simt_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
    const float* __restrict__ gamma, const float* __restrict__ omega,
    const float* __restrict__ phi, int H, int T, int64_t pos0, float eps,
    const float* __restrict__ S0, const float* __restrict__ z0, float* __restrict__ o,
    float* __restrict__ Dout, float* __restrict__ S_out, float* __restrict__ z_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem& sm = *reinterpret_cast<SimtSmem*>(smem_raw);
  const int bh = blockIdx.x;
  const int h = bh % H;
  const int tid = threadIdx.x;
  const int64_t seq = static_cast<int64_t>(bh) * T;
  const float g = gamma[h];

  for (int i = tid; i < kF * kDv; i += kThreads)
    sm.S[i] = S0 ? S0[static_cast<int64_t>(bh) * kF * kDv + i] : 0.f;
  for (int i = tid; i < kF; i += kThreads) sm.z[i] = z0 ? z0[static_cast<int64_t>(bh) * kF + i] : 0.f;

  for (int c0 = 0; c0 < T; c0 += kC) {
    const int nc = min(kC, T - c0);
    __syncthreads();  // previous chunk finished with pq, pk, v, P
    // Features of the chunk's queries and keys; rows past the end are zero.
    for (int e = tid; e < 2 * kC * kD; e += kThreads) {
      const int which = e / (kC * kD);
      const int t = (e / kD) % kC;
      const int a = e % kD;
      float* dst = (which == 0 ? sm.pq : sm.pk) + t * kFP + 6 * a;
      if (t < nc) {
        const Tin* src = which == 0 ? q : k;
        const float u = load_as_float(src + (seq + c0 + t) * kD + a);
        const float ph = phase_mod_2pi(pos0 + c0 + t, phi[h * kD + a]);
        const FeatAngles f = feat_exact(u, g, omega[h * kD + a], ph);
        float ch[6];
        feat_channels(f, ch);
#pragma unroll
        for (int cc = 0; cc < 6; ++cc) dst[cc] = ch[cc];
      } else {
#pragma unroll
        for (int cc = 0; cc < 6; ++cc) dst[cc] = 0.f;
      }
    }
    for (int e = tid; e < kC * kDv; e += kThreads) {
      const int t = e / kDv;
      sm.v[e] = t < nc ? load_as_float(v + (seq + c0 + t) * kDv + (e % kDv)) : 0.f;
    }
    __syncthreads();

    // Masked intra-chunk scores P[t][j], j <= t.
    {
      const int t = tid >> 3;
      const float* rq = sm.pq + t * kFP;
#pragma unroll
      for (int m = 0; m < kC / 8; ++m) {
        const int j = (tid & 7) + 8 * m;
        float s = 0.f;
        if (j <= t) {
          const float* rk = sm.pk + j * kFP;
          for (int f = 0; f < kF; ++f) s = fmaf(rq[f], rk[f], s);
        }
        sm.P[t * (kC + 1) + j] = s;
      }
    }
    __syncthreads();

    // Numerator and denominator of every query row; write o and D.
    {
      const int t = tid >> 3;
      const int lane8 = tid & 7;
      const float* rq = sm.pq + t * kFP;
      float num[kDv / 8];
#pragma unroll
      for (int m = 0; m < kDv / 8; ++m) num[m] = 0.f;
      for (int j = 0; j <= t; ++j) {
        const float p = sm.P[t * (kC + 1) + j];
#pragma unroll
        for (int m = 0; m < kDv / 8; ++m) num[m] = fmaf(p, sm.v[j * kDv + lane8 + 8 * m], num[m]);
      }
      for (int f = 0; f < kF; ++f) {
        const float x = rq[f];
#pragma unroll
        for (int m = 0; m < kDv / 8; ++m) num[m] = fmaf(x, sm.S[f * kDv + lane8 + 8 * m], num[m]);
      }
      float den = 0.f;
      for (int j = lane8; j <= t; j += 8) den += sm.P[t * (kC + 1) + j];
      for (int f = lane8; f < kF; f += 8) den = fmaf(rq[f], sm.z[f], den);
#pragma unroll
      for (int off = 4; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
      if (t < nc) {
        float* orow = o + (seq + c0 + t) * kDv;
        const float inv = 1.0f / (den + eps);
#pragma unroll
        for (int m = 0; m < kDv / 8; ++m) orow[lane8 + 8 * m] = num[m] * inv;
        if (Dout && lane8 == 0) Dout[seq + c0 + t] = den;
      }
    }
    __syncthreads();

    // State carry: S += Phi(K)^T V, z += column sums of Phi(K).
    {
      const int e = tid & (kDv - 1);
      for (int f = tid >> 6; f < kF; f += kThreads / kDv) {
        float acc = sm.S[f * kDv + e];
        for (int j = 0; j < nc; ++j) acc = fmaf(sm.pk[j * kFP + f], sm.v[j * kDv + e], acc);
        sm.S[f * kDv + e] = acc;
      }
      for (int f = tid; f < kF; f += kThreads) {
        float acc = sm.z[f];
        for (int j = 0; j < nc; ++j) acc += sm.pk[j * kFP + f];
        sm.z[f] = acc;
      }
    }
  }
  __syncthreads();
  if (S_out) {
    for (int i = tid; i < kF * kDv; i += kThreads) S_out[static_cast<int64_t>(bh) * kF * kDv + i] = sm.S[i];
    for (int i = tid; i < kF; i += kThreads) z_out[static_cast<int64_t>(bh) * kF + i] = sm.z[i];
  }
}

template <typename Tin>
cudaError_t launch(const ChunkFwdArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(SimtSmem);
  auto kern = chunk_fwd_simt_kernel<Tin>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const ProfileEvents& pe = profile_events();
  if (pe.start != nullptr) cudaEventRecord(pe.start, st);
  kern<<<a.B * a.H, kThreads, smem, st>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v),
      a.gamma, a.omega, a.phi, a.H, a.T, a.pos0, a.eps, a.S0, a.z0, a.o, a.D, a.S_out, a.z_out);
  e = cudaGetLastError();
  if (pe.stop != nullptr) cudaEventRecord(pe.stop, st);
  return e;
}

}  // namespace

size_t chunk_fwd_simt_smem_bytes() { return sizeof(SimtSmem); }

cudaError_t chunk_fwd_simt_launch(const ChunkFwdArgs& a, cudaStream_t st) {
  if (a.B * a.H == 0) return cudaSuccess;
  return a.in_dtype == SANATAN_F32 ? launch<float>(a, st) : launch<__nv_bfloat16>(a, st);
}

}  // namespace sanatan
