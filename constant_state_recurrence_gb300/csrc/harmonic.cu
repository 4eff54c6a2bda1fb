// The harmonic feature map of the reading notes' Appendix B ("附录 B 的频谱展望"):
// cos(n theta), sin(n theta) for n = 1..N added to the angle block, which keeps
// the p = 1 attention an explicit feature-map attention with a constant-size
// state (larger by the number of harmonics).  Per dimension a the features are
//   [A, r A],  A = [1, cos th, sin th, cos 2th, sin 2th, ..., cos N th, sin N th],
// th the rotated angle of eq. (4) and r the soft root of eq. (3) from the
// un-rotated angle; channel l (2N + 1) + m of dimension a sits at
// a * 2(2N + 1) + l (2N + 1) + m (N = 1 is the six-channel map of eq. (6)).
// The kernel per dimension is (1 + r_q r_k)(1 + sum_n cos(n dtheta)).
//
// Three kernels, all float32 on the CUDA cores: the elementwise feature map,
// the chunked causal forward (one CTA per sequence, the state in shared
// memory, chunks of 8 tokens; N = 1 is the six-channel f32 path), and the decode step
// (a cluster of 4 CTAs per slot splitting the state rows).
#include <cooperative_groups.h>

#include "sanatan_internal.h"
#include "sanatan_math.cuh"

namespace sanatan {
namespace {

namespace cg = cooperative_groups;

constexpr int kD = 64;
constexpr int kDv = 64;

template <int N>
struct Harm {
  static constexpr int kAng = 2 * N + 1;   // angle block
  static constexpr int kCh = 2 * kAng;     // channels per dimension
  static constexpr int kF = kCh * kD;      // features
};

// All channels of one dimension from u (float32, libm-grade sin/cos/tanh);
// the multiples of the rotated angle by the angle-addition recurrence.
template <int N>
__device__ __forceinline__ void harmonic_channels(float u, float gamma, float omega, float phase,
                                                  float (&ch)[Harm<N>::kCh]) {
  const FeatAngles f = feat_exact(u, gamma, omega, phase);   // cos, sin of th_rot; r
  constexpr int kA = Harm<N>::kAng;
  float c = f.c, s = f.s;
  ch[0] = 1.0f;
  ch[1] = c;
  ch[2] = s;
#pragma unroll
  for (int n = 2; n <= N; ++n) {
    const float cn = fmaf(c, f.c, -s * f.s);
    const float sn = fmaf(s, f.c, c * f.s);
    c = cn;
    s = sn;
    ch[2 * n - 1] = c;
    ch[2 * n] = s;
  }
#pragma unroll
  for (int m = 0; m < kA; ++m) ch[kA + m] = f.r * ch[m];
}

template <int N, typename Tin, typename Tout>
__global__ void __launch_bounds__(256) featurize_harmonic_kernel(
    const Tin* __restrict__ u, const float* __restrict__ gamma, const float* __restrict__ omega,
    const float* __restrict__ phi, Tout* __restrict__ out, int H, int T, int64_t pos0,
    int64_t total) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int a = static_cast<int>(idx % kD);
  const int64_t row = idx / kD;
  const int i = static_cast<int>(row % T);
  const int h = static_cast<int>((row / T) % H);
  float ch[Harm<N>::kCh];
  harmonic_channels<N>(load_as_float(u + idx), gamma[h], omega[h * kD + a],
                       phase_mod_2pi(pos0 + i, phi[h * kD + a]), ch);
  Tout* dst = out + idx * Harm<N>::kCh;
#pragma unroll
  for (int c = 0; c < Harm<N>::kCh; ++c) dst[c] = store_from_float<Tout>(ch[c]);
}

// ---------------------------------------------------------------------------
// Chunked forward (N = 2): per chunk of kC = 8 tokens, the masked scores from
// the chunk's features, the outputs from them plus Phi(q) against the state of
// the earlier chunks, then S += Phi(K)^T V, z += Phi(K)^T 1.
constexpr int kThreads = 256;

template <int N, int C>
struct HarmSmem {
  static constexpr int kF = Harm<N>::kF;
  static constexpr int kFP = kF + 1;   // padded row stride
  float pq[C * kFP];
  float pk[C * kFP];
  float v[C * kDv];
  float S[kF * kDv];
  float z[kF];
  float P[C * (C + 1)];
};

template <int N, int C, typename Tin>
__global__ void __launch_bounds__(kThreads, 1) chunk_fwd_harmonic_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
    const float* __restrict__ gamma, const float* __restrict__ omega,
    const float* __restrict__ phi, int H, int T, int64_t pos0, float eps,
    const float* __restrict__ S0, const float* __restrict__ z0, float* __restrict__ o,
    float* __restrict__ Dout, float* __restrict__ S_out, float* __restrict__ z_out) {
  using Sm = HarmSmem<N, C>;
  constexpr int kF = Sm::kF, kFP = Sm::kFP, kCh = Harm<N>::kCh;
  constexpr int kPairLanes = kThreads / (C * C);   // threads per (t, j) score
  constexpr int kRowLanes = kThreads / C;          // threads per output row
  static_assert(kPairLanes >= 1 && (kPairLanes & (kPairLanes - 1)) == 0 && kRowLanes <= 32,
                "thread mapping");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Sm& sm = *reinterpret_cast<Sm*>(smem_raw);
  const int bh = blockIdx.x;
  const int h = bh % H;
  const int tid = threadIdx.x;
  const int64_t seq = static_cast<int64_t>(bh) * T;
  const float g = gamma[h];

  for (int i = tid; i < kF * kDv; i += kThreads)
    sm.S[i] = S0 ? S0[static_cast<int64_t>(bh) * kF * kDv + i] : 0.f;
  for (int i = tid; i < kF; i += kThreads) sm.z[i] = z0 ? z0[static_cast<int64_t>(bh) * kF + i] : 0.f;

  for (int c0 = 0; c0 < T; c0 += C) {
    const int nc = min(C, T - c0);
    __syncthreads();  // the previous chunk is done with pq, pk, v, P and S
    for (int e = tid; e < 2 * C * kD; e += kThreads) {
      const int which = e / (C * kD);
      const int t = (e / kD) % C;
      const int a = e % kD;
      float* dst = (which == 0 ? sm.pq : sm.pk) + t * kFP + kCh * a;
      if (t < nc) {
        const Tin* src = which == 0 ? q : k;
        float ch[kCh];
        harmonic_channels<N>(load_as_float(src + (seq + c0 + t) * kD + a), g, omega[h * kD + a],
                             phase_mod_2pi(pos0 + c0 + t, phi[h * kD + a]), ch);
#pragma unroll
        for (int cc = 0; cc < kCh; ++cc) dst[cc] = ch[cc];
      } else {
#pragma unroll
        for (int cc = 0; cc < kCh; ++cc) dst[cc] = 0.f;
      }
    }
    for (int e = tid; e < C * kDv; e += kThreads) {
      const int t = e / kDv;
      sm.v[e] = t < nc ? load_as_float(v + (seq + c0 + t) * kDv + (e % kDv)) : 0.f;
    }
    __syncthreads();

    // masked scores P[t][j], j <= t: kPairLanes threads per pair
    {
      const int pair = tid / kPairLanes, part = tid % kPairLanes;
      const int t = pair / C, j = pair % C;
      float s = 0.f;
      if (j <= t) {
        const float* rq = sm.pq + t * kFP;
        const float* rk = sm.pk + j * kFP;
        for (int f = part; f < kF; f += kPairLanes) s = fmaf(rq[f], rk[f], s);
      }
#pragma unroll
      for (int off = kPairLanes / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (part == 0) sm.P[t * (C + 1) + j] = s;
    }
    __syncthreads();

    // outputs: kRowLanes threads per row, kDv / kRowLanes columns each
    {
      constexpr int kCols = kDv / kRowLanes;
      const int t = tid / kRowLanes, lane = tid % kRowLanes;
      const float* rq = sm.pq + t * kFP;
      float num[kCols];
#pragma unroll
      for (int m = 0; m < kCols; ++m) num[m] = 0.f;
      for (int j = 0; j <= t; ++j) {
        const float p = sm.P[t * (C + 1) + j];
#pragma unroll
        for (int m = 0; m < kCols; ++m) num[m] = fmaf(p, sm.v[j * kDv + lane + kRowLanes * m], num[m]);
      }
      for (int f = 0; f < kF; ++f) {
        const float x = rq[f];
#pragma unroll
        for (int m = 0; m < kCols; ++m) num[m] = fmaf(x, sm.S[f * kDv + lane + kRowLanes * m], num[m]);
      }
      float den = 0.f;
      for (int j = lane; j <= t; j += kRowLanes) den += sm.P[t * (C + 1) + j];
      for (int f = lane; f < kF; f += kRowLanes) den = fmaf(rq[f], sm.z[f], den);
#pragma unroll
      for (int off = kRowLanes / 2; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
      if (t < nc) {
        float* orow = o + (seq + c0 + t) * kDv;
        const float inv = 1.0f / (den + eps);
#pragma unroll
        for (int m = 0; m < kCols; ++m) orow[lane + kRowLanes * m] = num[m] * inv;
        if (Dout && lane == 0) Dout[seq + c0 + t] = den;
      }
    }
    __syncthreads();

    // state carry
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

// ---------------------------------------------------------------------------
// Decode step with the harmonic map: a cluster of R CTAs per slot, each with
// kF / R feature rows (whole dimensions), as the six-channel decode kernel.
template <int N, int R, int T>
__global__ void __launch_bounds__(T) decode_harmonic_kernel(
    float* __restrict__ S, float* __restrict__ z, const float* __restrict__ q,
    const float* __restrict__ k, const float* __restrict__ v, const float* __restrict__ gamma,
    const float* __restrict__ omega, const float* __restrict__ phi,
    const int64_t* __restrict__ pos, int G, float eps, float* __restrict__ o) {
  constexpr int kCh = Harm<N>::kCh, kF = Harm<N>::kF;
  constexpr int kColGroups = kDv / 4;
  constexpr int kRows = kF / R;
  constexpr int kDims = kD / R;
  constexpr int kRowLanes = T / kColGroups;
  constexpr int kPer = kRows / kRowLanes;
  static_assert(kRows % kRowLanes == 0 && kDims * kCh == kRows && 2 * kDims + kDv <= T, "shape");
  __shared__ float s_fq[kRows];
  __shared__ float s_fk[kRows];
  __shared__ __align__(16) float s_v[kDv];
  __shared__ float s_num[kRowLanes / 2][kDv + 4];
  __shared__ float s_part[kDv + 1];
  __shared__ float s_den[T / 32];

  const int rank = static_cast<int>(cg::this_cluster().block_rank());
  const int n = blockIdx.x / R;
  const int g = n % G;
  const int tid = threadIdx.x;
  const int row0 = rank * kRows;
  const int cgp = tid % kColGroups;
  const int r0 = tid / kColGroups;
  float4* Sn = reinterpret_cast<float4*>(S + (static_cast<int64_t>(n) * kF + row0) * kDv);
  float4 x[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) x[i] = Sn[(r0 + i * kRowLanes) * kColGroups + cgp];
  float* zn = z + static_cast<int64_t>(n) * kF + row0;
  constexpr int kZ = (kRows + T - 1) / T;
  float zr[kZ];
#pragma unroll
  for (int i = 0; i < kZ; ++i) {
    const int f = tid + i * T;
    zr[i] = f < kRows ? zn[f] : 0.f;
  }
  if (tid < 2 * kDims) {
    const int a = rank * kDims + (tid % kDims);
    const float u = (tid < kDims ? q : k)[static_cast<int64_t>(n) * kD + a];
    float ch[kCh];
    harmonic_channels<N>(u, gamma[g], omega[g * kD + a], phase_mod_2pi(pos[n], phi[g * kD + a]), ch);
    float* dst = (tid < kDims ? s_fq : s_fk) + kCh * (tid % kDims);
#pragma unroll
    for (int c = 0; c < kCh; ++c) dst[c] = ch[c];
  } else if (tid < 2 * kDims + kDv) {
    s_v[tid - 2 * kDims] = v[static_cast<int64_t>(n) * kDv + (tid - 2 * kDims)];
  }
  __syncthreads();
  const float4 vv = reinterpret_cast<const float4*>(s_v)[cgp];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int r = r0 + i * kRowLanes;
    const float pk = s_fk[r];
    float4 y = x[i];
    y.x = fmaf(pk, vv.x, y.x);
    y.y = fmaf(pk, vv.y, y.y);
    y.z = fmaf(pk, vv.z, y.z);
    y.w = fmaf(pk, vv.w, y.w);
    Sn[r * kColGroups + cgp] = y;
    const float pq = s_fq[r];
    acc.x = fmaf(pq, y.x, acc.x);
    acc.y = fmaf(pq, y.y, acc.y);
    acc.z = fmaf(pq, y.z, acc.z);
    acc.w = fmaf(pq, y.w, acc.w);
  }
  acc.x += __shfl_xor_sync(0xffffffffu, acc.x, 16);
  acc.y += __shfl_xor_sync(0xffffffffu, acc.y, 16);
  acc.z += __shfl_xor_sync(0xffffffffu, acc.z, 16);
  acc.w += __shfl_xor_sync(0xffffffffu, acc.w, 16);
  if ((tid & 16) == 0) {
    float* dst = &s_num[r0 >> 1][4 * cgp];
    dst[0] = acc.x;
    dst[1] = acc.y;
    dst[2] = acc.z;
    dst[3] = acc.w;
  }
  float den = 0.f;
#pragma unroll
  for (int i = 0; i < kZ; ++i) {
    const int f = tid + i * T;
    if (f < kRows) {
      const float zz = zr[i] + s_fk[f];
      zn[f] = zz;
      den = fmaf(s_fq[f], zz, den);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  if ((tid & 31) == 0) s_den[tid >> 5] = den;
  __syncthreads();
  if (tid < kDv) {
    float num = 0.f;
#pragma unroll
    for (int i = 0; i < kRowLanes / 2; ++i) num += s_num[i][tid];
    s_part[tid] = num;
  } else if (tid == kDv) {
    float dsum = 0.f;
#pragma unroll
    for (int w = 0; w < T / 32; ++w) dsum += s_den[w];
    s_part[kDv] = dsum;
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();  // every CTA's partial sums are in its shared memory
  if (rank == 0 && tid < kDv) {
    float num = 0.f, dsum = 0.f;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      const float* part = cluster.map_shared_rank(s_part, rr);
      num += part[tid];
      dsum += part[kDv];
    }
    o[static_cast<int64_t>(n) * kDv + tid] = num / (dsum + eps);
  }
  cluster.sync();  // no CTA leaves while rank 0 still reads its shared memory
}

template <int N, typename Tin, typename Tout>
cudaError_t featurize_h(const HarmonicFeatArgs& a, cudaStream_t st) {
  const int64_t total = static_cast<int64_t>(a.B) * a.H * a.T * kD;
  if (total == 0) return cudaSuccess;
  featurize_harmonic_kernel<N, Tin, Tout><<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(
      static_cast<const Tin*>(a.u), a.gamma, a.omega, a.phi, static_cast<Tout*>(a.out), a.H, a.T,
      a.pos0, total);
  return cudaGetLastError();
}

template <int N>
cudaError_t featurize_n(const HarmonicFeatArgs& a, cudaStream_t st) {
  if (a.u_dtype == SANATAN_F32 && a.out_dtype == SANATAN_F32) return featurize_h<N, float, float>(a, st);
  if (a.u_dtype == SANATAN_F32) return featurize_h<N, float, __nv_bfloat16>(a, st);
  if (a.out_dtype == SANATAN_F32) return featurize_h<N, __nv_bfloat16, float>(a, st);
  return featurize_h<N, __nv_bfloat16, __nv_bfloat16>(a, st);
}

template <int N, int C, typename Tin>
cudaError_t chunk_h(const ChunkFwdArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(HarmSmem<N, C>);
  auto kern = chunk_fwd_harmonic_kernel<N, C, Tin>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<a.B * a.H, kThreads, smem, st>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v),
      a.gamma, a.omega, a.phi, a.H, a.T, a.pos0, a.eps, a.S0, a.z0, a.o, a.D, a.S_out, a.z_out);
  return cudaGetLastError();
}

template <int N>
cudaError_t decode_h(float* S, float* z, const float* q, const float* k, const float* v,
                     const float* gamma, const float* omega, const float* phi,
                     const int64_t* pos, int Nslots, int G, float eps, float* o,
                     cudaStream_t st) {
  constexpr int kR = 4;
  constexpr int kT = 256;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(Nslots) * kR);
  cfg.blockDim = dim3(kT);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kR;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_harmonic_kernel<N, kR, kT>, S, z, q, k, v, gamma, omega,
                            phi, pos, G, eps, o);
}

}  // namespace

cudaError_t featurize_harmonic_launch(const HarmonicFeatArgs& a, cudaStream_t st) {
  switch (a.harmonics) {
    case 1: return featurize_n<1>(a, st);
    case 2: return featurize_n<2>(a, st);
    case 3: return featurize_n<3>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t chunk_fwd_harmonic_launch(const ChunkFwdArgs& a, int harmonics, cudaStream_t st) {
  if (a.B * a.H == 0) return cudaSuccess;
  const bool f32 = a.in_dtype == SANATAN_F32;
  if (harmonics == 1) return chunk_fwd_simt_launch(a, st);  // the six-channel map itself
  if (harmonics == 2) return f32 ? chunk_h<2, 8, float>(a, st) : chunk_h<2, 8, __nv_bfloat16>(a, st);
  return cudaErrorInvalidValue;
}

cudaError_t decode_harmonic_launch(float* S, float* z, const float* q, const float* k,
                                   const float* v, const float* gamma, const float* omega,
                                   const float* phi, const int64_t* pos, int N, int G, float eps,
                                   int harmonics, float* o, cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  switch (harmonics) {
    case 1: return decode_h<1>(S, z, q, k, v, gamma, omega, phi, pos, N, G, eps, o, st);
    case 2: return decode_h<2>(S, z, q, k, v, gamma, omega, phi, pos, N, G, eps, o, st);
    case 3: return decode_h<3>(S, z, q, k, v, gamma, omega, phi, pos, N, G, eps, o, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sanatan
