// One decode token of the constant-state recurrence (reading notes §2.7,
// paper eq. (9)) for N independent state slots, in place:
//   S <- S + Phi(k) v^T,  z <- z + Phi(k),  o = Phi(q)^T S / (Phi(q)^T z + eps).
// The step streams each slot's 6d x dv float32 state once (read + write); the
// readout is reduced with warp shuffles and a small shared-memory tree.
#include "sanatan_internal.h"
#include "sanatan_math.cuh"

namespace sanatan {
namespace {

constexpr int kD = 64;
constexpr int kDv = 64;
constexpr int kF = 6 * kD;            // 384 feature rows
constexpr int kThreads = 256;
constexpr int kColGroups = kDv / 4;   // 16 float4 column groups per row
constexpr int kRowLanes = kThreads / kColGroups;  // 16 rows in flight per pass

__global__ void __launch_bounds__(kThreads) decode_step_kernel(
    float* __restrict__ S, float* __restrict__ z, const float* __restrict__ q,
    const float* __restrict__ k, const float* __restrict__ v, const float* __restrict__ gamma,
    const float* __restrict__ omega, const float* __restrict__ phi,
    const int64_t* __restrict__ pos, int G, float eps, float* __restrict__ o) {
  __shared__ float s_fq[kF];
  __shared__ float s_fk[kF];
  __shared__ __align__(16) float s_v[kDv];
  __shared__ float s_num[kRowLanes][kDv + 4];
  __shared__ float s_den[kThreads / 32];

  const int n = blockIdx.x;
  const int g = n % G;
  const int tid = threadIdx.x;

  // Features of this slot's q (threads 0..63) and k (64..127); v (128..191).
  if (tid < 2 * kD) {
    const int a = tid & (kD - 1);
    const float u = (tid < kD ? q : k)[static_cast<int64_t>(n) * kD + a];
    const float ph = phase_mod_2pi(pos[n], phi[g * kD + a]);
    const FeatAngles f = feat_exact(u, gamma[g], omega[g * kD + a], ph);
    float ch[6];
    feat_channels(f, ch);
    float* dst = (tid < kD ? s_fq : s_fk) + 6 * a;
#pragma unroll
    for (int c = 0; c < 6; ++c) dst[c] = ch[c];
  } else if (tid < 2 * kD + kDv) {
    s_v[tid - 2 * kD] = v[static_cast<int64_t>(n) * kDv + (tid - 2 * kD)];
  }
  __syncthreads();

  // S rows: thread (row lane r0, column group cg) walks rows r0, r0+16, ...
  const int cg = tid % kColGroups;
  const int r0 = tid / kColGroups;
  const float4 vv = reinterpret_cast<const float4*>(s_v)[cg];
  float4* Sn = reinterpret_cast<float4*>(S + static_cast<int64_t>(n) * kF * kDv);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int r = r0; r < kF; r += kRowLanes) {
    float4 x = Sn[r * kColGroups + cg];
    const float pk = s_fk[r];
    x.x = fmaf(pk, vv.x, x.x);
    x.y = fmaf(pk, vv.y, x.y);
    x.z = fmaf(pk, vv.z, x.z);
    x.w = fmaf(pk, vv.w, x.w);
    Sn[r * kColGroups + cg] = x;
    const float pq = s_fq[r];
    acc.x = fmaf(pq, x.x, acc.x);
    acc.y = fmaf(pq, x.y, acc.y);
    acc.z = fmaf(pq, x.z, acc.z);
    acc.w = fmaf(pq, x.w, acc.w);
  }
  // Two row lanes share a warp (lanes l and l+16 have the same column group).
  acc.x += __shfl_xor_sync(0xffffffffu, acc.x, 16);
  acc.y += __shfl_xor_sync(0xffffffffu, acc.y, 16);
  acc.z += __shfl_xor_sync(0xffffffffu, acc.z, 16);
  acc.w += __shfl_xor_sync(0xffffffffu, acc.w, 16);
  if ((tid & 16) == 0) {
    float* dst = &s_num[r0 >> 1][4 * cg];
    dst[0] = acc.x;
    dst[1] = acc.y;
    dst[2] = acc.z;
    dst[3] = acc.w;
  }

  // z rows and the denominator.
  float den = 0.f;
  float* zn = z + static_cast<int64_t>(n) * kF;
  for (int f = tid; f < kF; f += kThreads) {
    const float zz = zn[f] + s_fk[f];
    zn[f] = zz;
    den = fmaf(s_fq[f], zz, den);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  if ((tid & 31) == 0) s_den[tid >> 5] = den;
  __syncthreads();

  if (tid < kDv) {
    float num = 0.f;
#pragma unroll
    for (int i = 0; i < kRowLanes / 2; ++i) num += s_num[i][tid];
    float dsum = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) dsum += s_den[w];
    o[static_cast<int64_t>(n) * kDv + tid] = num / (dsum + eps);
  }
}

}  // namespace

cudaError_t decode_step_launch(float* S, float* z, const float* q, const float* k,
                               const float* v, const float* gamma, const float* omega,
                               const float* phi, const int64_t* pos, int N, int G, float eps,
                               float* o, cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  decode_step_kernel<<<N, kThreads, 0, st>>>(S, z, q, k, v, gamma, omega, phi, pos, G, eps, o);
  return cudaGetLastError();
}

}  // namespace sanatan
