// One decode token of the constant-state recurrence (reading notes §2.7,
// paper eq. (9)) for N independent state slots, in place:
//   S <- S + Phi(k) v^T,  z <- z + Phi(k),  o = Phi(q)^T S / (Phi(q)^T z + eps).
// The step streams each slot's 6d x dv float32 state once (read + write).
//
// A slot is handled by one CTA (1024 threads when there are at most two slots
// per SM, 256 when there are more than four) or split over a cluster of R
// CTAs by feature rows (R = 4 in between, R = 8 when there are at most one
// slot per eight SMs).  Each CTA issues the loads of
// its whole row block first and featurises q and k for its rows while they
// are in flight; the readout partial sums (numerator and denominator) are
// reduced with warp shuffles, a shared-memory tree and, across the cluster,
// distributed shared memory read by CTA rank 0.
#include <cooperative_groups.h>

#include "sanatan_internal.h"
#include "decode_math.cuh"
#include "sanatan_math.cuh"

namespace sanatan {
namespace {

namespace cg = cooperative_groups;

constexpr int kD = 64;
constexpr int kDv = 64;
constexpr int kF = 6 * kD;            // 384 feature rows
constexpr int kColGroups = kDv / 4;   // 16 float4 column groups per row

using decm::feat_decode;

template <int R, int T>
__global__ void __launch_bounds__(T) decode_step_kernel(
    float* __restrict__ S, float* __restrict__ z, const float* __restrict__ q,
    const float* __restrict__ k, const float* __restrict__ v, const float* __restrict__ gamma,
    const float* __restrict__ omega, const float* __restrict__ phi,
    const int64_t* __restrict__ pos, int G, float eps, float* __restrict__ o) {
  constexpr int kRows = kF / R;             // feature rows of this CTA
  constexpr int kDims = kD / R;             // dimensions of this CTA (6 rows each)
  constexpr int kRowLanes = T / kColGroups;
  constexpr int kPer = kRows / kRowLanes;   // float4 of S per thread
  static_assert(kRows % kRowLanes == 0 && kDims * 6 == kRows && 2 * kDims + kDv <= T, "shape");
  __shared__ float s_fq[kRows];
  __shared__ float s_fk[kRows];
  __shared__ __align__(16) float s_v[kDv];
  __shared__ float s_num[kRowLanes / 2][kDv + 4];
  __shared__ float s_part[kDv + 1];
  __shared__ float s_den[T / 32];

  const int rank = (R > 1) ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
  const int n = blockIdx.x / R;
  const int g = n % G;
  const int tid = threadIdx.x;
  const int row0 = rank * kRows;  // first feature row of this CTA

  // Loads of this CTA's S rows and z rows, issued before anything else.
  const int cgp = tid % kColGroups;
  const int r0 = tid / kColGroups;
  float4* Sn = reinterpret_cast<float4*>(S + (static_cast<int64_t>(n) * kF + row0) * kDv);
  float4 x[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) x[i] = Sn[(r0 + i * kRowLanes) * kColGroups + cgp];
  float* zn = z + static_cast<int64_t>(n) * kF + row0;
  float zr[(kRows + T - 1) / T];
#pragma unroll
  for (int i = 0; i < (kRows + T - 1) / T; ++i) {
    const int f = tid + i * T;
    zr[i] = f < kRows ? zn[f] : 0.f;
  }

  // Features of this CTA's dimensions of q (threads 0..kDims-1) and k
  // (kDims..2kDims-1); v (next 64 threads).
  if (tid < 2 * kDims) {
    const int a = rank * kDims + (tid % kDims);
    const float u = (tid < kDims ? q : k)[static_cast<int64_t>(n) * kD + a];
    const float ph = phase_mod_2pi(pos[n], phi[g * kD + a]);
    float ch[6];
    feat_decode(u, gamma[g], omega[g * kD + a], ph, ch);
    float* dst = (tid < kDims ? s_fq : s_fk) + 6 * (tid % kDims);
#pragma unroll
    for (int c = 0; c < 6; ++c) dst[c] = ch[c];
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
  // Lanes l and l+16 of a warp have the same column group.
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

  // z rows and the denominator.
  float den = 0.f;
#pragma unroll
  for (int i = 0; i < (kRows + T - 1) / T; ++i) {
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
  if constexpr (R > 1) {
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
  } else {
    __syncthreads();
    if (tid < kDv) o[static_cast<int64_t>(n) * kDv + tid] = s_part[tid] / (s_part[kDv] + eps);
  }
}

int sm_count_decode() {
  static int cached = 0;
  if (cached == 0) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      cached = n;
    else
      return 152;
  }
  return cached;
}

// One slot per cluster of R CTAs of 128 threads (rows split by CTA rank).
template <int R>
cudaError_t launch_cluster(float* S, float* z, const float* q, const float* k, const float* v,
                           const float* gamma, const float* omega, const float* phi,
                           const int64_t* pos, int N, int G, float eps, float* o, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(N) * R);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = R;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_step_kernel<R, 128>, S, z, q, k, v, gamma, omega, phi,
                            pos, G, eps, o);
}

}  // namespace

cudaError_t decode_step_launch(float* S, float* z, const float* q, const float* k,
                               const float* v, const float* gamma, const float* omega,
                               const float* phi, const int64_t* pos, int N, int G, float eps,
                               float* o, cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  // At most one slot per eight SMs (the layers of a batch-1 stack step): an
  // 8-CTA cluster per slot, so that many SMs stream each slot's state.
  if (8LL * N <= sm_count_decode())
    return launch_cluster<8>(S, z, q, k, v, gamma, omega, phi, pos, N, G, eps, o, st);
  // Up to two slots per SM: one 1024-thread CTA per slot (six state loads in
  // flight per thread); up to four: a 4-CTA cluster per slot so that every SM
  // streams part of the state; more: one 256-thread CTA per slot.
  if (static_cast<int64_t>(N) <= 2LL * sm_count_decode()) {
    decode_step_kernel<1, 1024><<<N, 1024, 0, st>>>(S, z, q, k, v, gamma, omega, phi, pos, G, eps,
                                                    o);
    return cudaGetLastError();
  }
  if (static_cast<int64_t>(N) < 4LL * sm_count_decode())
    return launch_cluster<4>(S, z, q, k, v, gamma, omega, phi, pos, N, G, eps, o, st);
  decode_step_kernel<1, 256><<<N, 256, 0, st>>>(S, z, q, k, v, gamma, omega, phi, pos, G, eps, o);
  return cudaGetLastError();
}

}  // namespace sanatan
