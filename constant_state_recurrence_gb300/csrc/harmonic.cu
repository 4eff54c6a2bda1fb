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
// Kernels, all float32 on the CUDA cores: the elementwise feature map; the
// chunked causal forward (a cluster of 8 CTAs per sequence, each holding the
// state rows of 8 dimensions in registers; N = 1 is the six-channel f32 path);
// its backward (a preparation kernel, the forward recurrence in reverse time for
// dv, and the feature-space passes for dq and dk with the chain rule); and the
// decode step (a cluster of 4 CTAs per slot splitting the state rows).
#include <cooperative_groups.h>

#include "sanatan_internal.h"
#include "sanatan_math.cuh"
#include "f32x2.cuh"

namespace sanatan {
namespace {

namespace cg = cooperative_groups;
using f2::ffma2;
using f2::pk2;
using f2::upk2;

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
// Chunked forward: a cluster of kRanks CTAs per sequence, CTA rank r holding
// the state rows of dimensions 8r .. 8r + 7 (8 kCh rows x 64 columns) in
// registers.  Scores, the intra-chunk weighted values and the state readout
// are all sums over features, so per chunk of kCT tokens every CTA forms
// complete partial numerators and denominators from its own rows:
//   num_t = sum_{j<=t} (Phi(q_t) . Phi(k_j))_r v_j + Phi(q_t)_r S_r,
//   den_t = sum_{j<=t} (Phi(q_t) . Phi(k_j))_r     + Phi(q_t)_r z_r,
// and one cluster reduction through distributed shared memory (CTA rank r
// sums tokens r and r + 8 over the cluster) gives o_t = num_t / (den_t + eps);
// then S_r += Phi(K)_r^T V, z_r += Phi(K)_r^T 1 in registers.  Thread
// (c, g) owns column c of the CTA's rows g kPT .. (g + 1) kPT - 1, read from
// shared memory as 16-byte row pieces and multiplied in packed f32x2 pairs.
constexpr int kThreads = 256;
constexpr int kRanks = 8;      // CTAs per sequence: 8 dimensions each
constexpr int kCT = 16;        // tokens per chunk (two per CTA in the reduction)

template <int N>
struct ClusterSmem {
  static constexpr int kR = 8 * Harm<N>::kCh;   // state rows of this CTA
  static constexpr int kRP = kR + 4;            // feature row pitch (16-byte rows)
  alignas(16) float pq[kCT][kRP];
  alignas(16) float pk[kCT][kRP];
  float v[kCT][kDv];
  float z[kR];
  float P[kCT][kCT + 1];
  float part[4][kCT][kDv];          // readout partials of the four row groups
  float out[2][kCT][kDv + 1];       // this CTA's partial numerators | denominator (by chunk parity)
};

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// kGrad: the value gradient of the backward, dv_j = sum_{t>=j} s_tj dN_t, as
// this same recurrence in reverse time (token u processed at step T-1-u, at its
// own position) with queries k, keys q, values dN and no normalisation; the
// output is written in Tout and D, S_out, z_out are not produced.
template <int N, typename Tin, typename Tv, typename Tout, bool kGrad>
__global__ void __launch_bounds__(kThreads, 3) chunk_fwd_harmonic_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tv* __restrict__ v,
    const float* __restrict__ gamma, const float* __restrict__ omega,
    const float* __restrict__ phi, int H, int T, int64_t pos0, float eps,
    const float* __restrict__ S0, const float* __restrict__ z0, Tout* __restrict__ o,
    float* __restrict__ Dout, float* __restrict__ S_out, float* __restrict__ z_out) {
  constexpr int kCh = Harm<N>::kCh, kF = Harm<N>::kF;
  constexpr int kR = ClusterSmem<N>::kR;
  constexpr int kPT = kR / 4;   // rows per thread
  constexpr int kP4 = kPT / 4;  // 16-byte pieces of them
  static_assert(kPT % 4 == 0 && kRanks * 8 == kD && 2 * kRanks == kCT, "shape");
  static_assert(kThreads == 2 * kCT * 8 && kThreads == 4 * kDv, "thread map");
  __shared__ ClusterSmem<N> sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int bh = blockIdx.x / kRanks;
  const int h = bh % H;
  const int tid = threadIdx.x;
  const int c = tid & (kDv - 1), rg = tid >> 6;
  const int64_t seq = static_cast<int64_t>(bh) * T;
  const int64_t row0 = static_cast<int64_t>(bh) * kF + rank * kR;   // first state row of the CTA
  const int f0 = rg * kPT;                                           // first row of the thread

  // feature thread map: (tensor, token, dimension of the CTA)
  const int fw = tid >> 7, ft = (tid >> 3) & (kCT - 1), fa = rank * 8 + (tid & 7);
  const Tin* fsrc = fw ? k : q;
  const float g = gamma[h], om = omega[h * kD + fa], ph = phi[h * kD + fa];

  uint64_t Sr[kPT / 2];   // rows f0 + 2i, f0 + 2i + 1 of column c
#pragma unroll
  for (int i = 0; i < kPT / 2; ++i) {
    const float a0 = S0 ? S0[(row0 + f0 + 2 * i) * kDv + c] : 0.f;
    const float a1 = S0 ? S0[(row0 + f0 + 2 * i + 1) * kDv + c] : 0.f;
    Sr[i] = pk2(a0, a1);
  }
  if (tid < kR) sm.z[tid] = z0 ? z0[row0 + tid] : 0.f;

  // inputs of the next chunk, held in registers while the current one runs
  // step i of the recurrence reads token row(i)
  auto row = [&](int i) -> int { return kGrad ? T - 1 - i : i; };
  float uf = 0.f, vr[4] = {0.f, 0.f, 0.f, 0.f};
  auto prefetch = [&](int c0n) {
    const int nn = min(kCT, T - c0n);
    uf = ft < nn ? load_as_float(fsrc + (seq + row(c0n + ft)) * kD + fa) : 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int t = rg + 4 * m;
      vr[m] = t < nn ? load_as_float(v + (seq + row(c0n + t)) * kDv + c) : 0.f;
    }
  };
  if (T > 0) prefetch(0);

  int buf = 0;
  for (int c0 = 0; c0 < T; c0 += kCT, buf ^= 1) {
    const int nc = min(kCT, T - c0);
    __syncthreads();   // the previous chunk is done with pq, pk, v and z
    {
      float* dst = (fw ? &sm.pk[ft][0] : &sm.pq[ft][0]) + kCh * (tid & 7);
      if (ft < nc) {
        float ch[kCh];
        harmonic_channels<N>(uf, g, om, phase_mod_2pi(pos0 + row(c0 + ft), ph), ch);
#pragma unroll
        for (int cc = 0; cc < kCh; ++cc) dst[cc] = ch[cc];
      } else {
#pragma unroll
        for (int cc = 0; cc < kCh; ++cc) dst[cc] = 0.f;
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) sm.v[rg + 4 * m][c] = vr[m];
    }
    if (c0 + kCT < T) prefetch(c0 + kCT);
    __syncthreads();
    {
      // partial scores over this CTA's rows: thread (t, j)
      const int t = tid >> 4, j = tid & (kCT - 1);
      if (j <= t) {
        const ulonglong2* a = reinterpret_cast<const ulonglong2*>(&sm.pq[t][0]);
        const ulonglong2* b = reinterpret_cast<const ulonglong2*>(&sm.pk[j][0]);
        uint64_t s0 = 0, s1 = 0;
#pragma unroll 4
        for (int i = 0; i < kR / 4; ++i) {
          const ulonglong2 x = a[i], y = b[i];
          s0 = ffma2(x.x, y.x, s0);
          s1 = ffma2(x.y, y.y, s1);
        }
        float p0, p1, p2, p3;
        upk2(s0, p0, p1);
        upk2(s1, p2, p3);
        sm.P[t][j] = (p0 + p1) + (p2 + p3);
      }
    }
#pragma unroll 1
    for (int th = 0; th < kCT; th += 8) {
      // readout partials of this thread's rows against the state before the chunk
      uint64_t num[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) num[t] = 0;
#pragma unroll
      for (int i = 0; i < kP4; ++i) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const ulonglong2 x = reinterpret_cast<const ulonglong2*>(&sm.pq[th + t][f0])[i];
          num[t] = ffma2(x.x, Sr[2 * i], num[t]);
          num[t] = ffma2(x.y, Sr[2 * i + 1], num[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        float x0, x1;
        upk2(num[t], x0, x1);
        sm.part[rg][th + t][c] = x0 + x1;
      }
    }
    __syncthreads();
    {
      // this CTA's partial numerators and denominators: warp w, tokens w and w + 8
      const int w = tid >> 5, lane = tid & 31;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int t = w + 8 * hh;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int col = lane + 32 * m;
          float acc = (sm.part[0][t][col] + sm.part[1][t][col]) +
                      (sm.part[2][t][col] + sm.part[3][t][col]);
          for (int j = 0; j <= t; ++j) acc = fmaf(sm.P[t][j], sm.v[j][col], acc);
          sm.out[buf][t][col] = acc;
        }
        float dn = (lane <= t) ? sm.P[t][lane] : 0.f;
        for (int f = lane; f < kR; f += 32) dn = fmaf(sm.pq[t][f], sm.z[f], dn);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dn += __shfl_xor_sync(0xffffffffu, dn, off);
        if (lane == 0) sm.out[buf][t][kDv] = dn;
      }
    }
    cluster_arrive();  // this CTA's partials of the chunk are written
    __syncthreads();   // z is read; the state may move on
#pragma unroll 4
    for (int j = 0; j < kCT; ++j) {
      const float vj = sm.v[j][c];
      const uint64_t vv = pk2(vj, vj);
#pragma unroll
      for (int i = 0; i < kP4; ++i) {
        const ulonglong2 x = reinterpret_cast<const ulonglong2*>(&sm.pk[j][f0])[i];   // zero past T
        Sr[2 * i] = ffma2(x.x, vv, Sr[2 * i]);
        Sr[2 * i + 1] = ffma2(x.y, vv, Sr[2 * i + 1]);
      }
    }
    if (tid < kR) {
      float acc = sm.z[tid];
#pragma unroll
      for (int j = 0; j < kCT; ++j) acc += sm.pk[j][tid];
      sm.z[tid] = acc;
    }
    cluster_wait();    // every CTA's partials of this chunk are in its shared memory
    {
      // tokens rank and rank + 8 of the chunk: the sums over the cluster
      const int t = rank + kRanks * (tid >> 6), e = tid & (kDv - 1);
      if (tid < 2 * kDv && t < nc) {
        float nm = 0.f, dn = 0.f;
#pragma unroll
        for (int rr = 0; rr < kRanks; ++rr) {
          const float* rem = cluster.map_shared_rank(&sm.out[buf][t][0], rr);
          nm += rem[e];
          dn += rem[kDv];
        }
        const int64_t orow = seq + row(c0 + t);
        if constexpr (kGrad) {
          o[orow * kDv + e] = store_from_float<Tout>(nm);
        } else {
          o[orow * kDv + e] = nm / (dn + eps);
          if (e == 0 && Dout) Dout[orow] = dn;
        }
      }
    }
  }
  __syncthreads();
  if (!kGrad && S_out) {
#pragma unroll
    for (int i = 0; i < kPT / 2; ++i) {
      float a0, a1;
      upk2(Sr[i], a0, a1);
      S_out[(row0 + f0 + 2 * i) * kDv + c] = a0;
      S_out[(row0 + f0 + 2 * i + 1) * kDv + c] = a1;
    }
    if (tid < kR) z_out[row0 + tid] = sm.z[tid];
  }
  cluster_arrive();    // no CTA leaves while another still reads its shared memory
  cluster_wait();
}

// ---------------------------------------------------------------------------
// Backward of the chunked forward (N >= 2).  With Dh_t = D_t + eps,
// dN_t = dO_t / Dh_t and dD_t = -(dO_t . o_t) / Dh_t:
//   dv_j       = sum_{t>=j} s_tj dN_t                       (the kGrad forward),
//   dPhi(q_t)  = [S_t | z_t] [dN_t | dD_t]   (S_t, z_t inclusive of t, from S0, z0),
//   dPhi(k_j)  = [G_j | g_j] [v_j | 1],      G_j = sum_{t>=j} Phi(q_t) dN_t^T,
//                                             g_j = sum_{t>=j} Phi(q_t) dD_t,
// then the chain rule through the harmonic map per (token, dimension).  The
// two feature gradients are attentions in feature space: a 65-wide query
// ([dN|dD] or [v|1]) reads a state of F rows x 65 columns, so every feature
// row's gradient is a reduction over the 65 columns only and a CTA that owns
// the rows of 8 dimensions finishes their chain rule on its own (no cluster).

constexpr int kPrepRows = 8;   // tokens (warps) per block of the preparation kernel

// dN [rows, 64] and dD [rows] from dO, o, D: one warp per token.
template <typename Tg>
__global__ void __launch_bounds__(256) harm_bwd_prep_kernel(const float* __restrict__ o,
                                                            const float* __restrict__ D,
                                                            const Tg* __restrict__ dO, float eps,
                                                            int64_t rows, float* __restrict__ dN,
                                                            float* __restrict__ dD) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * kPrepRows + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const float inv = 1.0f / (D[r] + eps);
  const float g0 = load_as_float(dO + r * kDv + lane), g1 = load_as_float(dO + r * kDv + lane + 32);
  float dot = g0 * o[r * kDv + lane] + g1 * o[r * kDv + lane + 32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  dN[r * kDv + lane] = g0 * inv;
  dN[r * kDv + lane + 32] = g1 * inv;
  if (lane == 0) dD[r] = -dot * inv;
}

// Gradient of one dimension's channels back to u and the per-head parameters.
struct HarmGrad {
  float du, dgamma, domega, dphi;
};

template <int N>
__device__ __forceinline__ HarmGrad harmonic_vjp(float u, float g, float om, float phase,
                                                 float tpos, const float* dch) {
  constexpr int kA = Harm<N>::kAng;
  const float th = squash_exact(u);
  float sx, cx;
  sincosf(th + om, &sx, &cx);
  const float gx = cx - sx;
  const float gpx = -sx - cx;
  const float r = tanhf(g * gx);
  float s1, c1;
  sincosf(th + phase, &s1, &c1);
  // A_0 = 1 contributes only to dr
  float dr = dch[kA];
  float dth = 0.f;
  float cn = c1, sn = s1;
#pragma unroll
  for (int n = 1; n <= N; ++n) {
    if (n > 1) {
      const float cm = fmaf(cn, c1, -sn * s1);
      const float sm = fmaf(sn, c1, cn * s1);
      cn = cm;
      sn = sm;
    }
    const float dAc = fmaf(r, dch[kA + 2 * n - 1], dch[2 * n - 1]);
    const float dAs = fmaf(r, dch[kA + 2 * n], dch[2 * n]);
    dr = fmaf(cn, dch[kA + 2 * n - 1], fmaf(sn, dch[kA + 2 * n], dr));
    dth = fmaf(static_cast<float>(n), fmaf(cn, dAs, -sn * dAc), dth);
  }
  const float dpre = dr * (1.0f - r * r);
  const float den = 1.0f + fabsf(u);
  HarmGrad e;
  e.du = fmaf(dpre * g, gpx, dth) * kPi / (den * den);
  e.dgamma = dpre * gx;
  e.domega = dpre * g * gpx;
  e.dphi = dth * tpos;
  return e;
}

constexpr int kFsaCT = 16;     // tokens per chunk
constexpr int kQP = 68;        // row pitch of the 65-wide query / key rows (16-byte rows)

template <int N>
struct FsaSmem {
  static constexpr int kR = 8 * Harm<N>::kCh;
  alignas(16) float qa[kFsaCT][kQP];        // query rows: [dN|dD] (dq pass) or [v|1] (dk pass)
  alignas(16) float kb[kFsaCT][kQP];        // key rows:   [v|1] or [dN|dD]
  float pv[kFsaCT][kR + 1];                 // value features Phi(k) or Phi(q) of the CTA's rows
  // state readout per column quarter; quarter 0 then holds the chunk's feature
  // gradient (each (t, f) is summed and rewritten by one thread)
  float part[4][kFsaCT][kR];
  float ds[kFsaCT][kFsaCT + 1];             // pair scores query . key (causal)
  float red[4][8][3];                       // parameter-gradient partials per warp
};

// One CTA per (sequence, 8 dimensions, pass): blockIdx.y = 0 gives dq (forward
// time, state from S0, z0), 1 gives dk (reverse time, state from zero).  Thread
// (cq, f) = (tid / kR, tid % kR) holds columns 16 cq .. 16 cq + 15 of state row f
// (and column 64, the ones / dD column, for cq = 3) as packed pairs, so the
// lanes of a warp share one column quarter and read the 65-wide rows as
// broadcasts; the four quarters' partial readouts meet in shared memory.
template <int N, typename Tin, bool kKeys>
__device__ __forceinline__ void fsa_pass(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
    const float* __restrict__ dN, const float* __restrict__ dD, const float* __restrict__ gamma,
    const float* __restrict__ omega, const float* __restrict__ phi, int H, int T, int64_t pos0,
    const float* __restrict__ S0, const float* __restrict__ z0, Tin* __restrict__ dout,
    float* __restrict__ dgamma, float* __restrict__ domega, float* __restrict__ dphi,
    FsaSmem<N>& sm) {
  constexpr int kCh = Harm<N>::kCh, kF = Harm<N>::kF;
  constexpr int kR = FsaSmem<N>::kR;
  const int grp = blockIdx.x & 7;              // dimensions 8 grp .. 8 grp + 7
  const int bh = blockIdx.x >> 3;
  const int h = bh % H;
  const int tid = threadIdx.x;
  const int f = tid % kR, cq = tid / kR;
  const int64_t seq = static_cast<int64_t>(bh) * T;
  const int64_t frow = static_cast<int64_t>(bh) * kF + grp * kR + f;   // global state row
  const float g = gamma[h];
  auto row = [&](int i) -> int { return kKeys ? T - 1 - i : i; };

  uint64_t W[8];
  float w64 = 0.f;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    float a0 = 0.f, a1 = 0.f;
    if (!kKeys && S0) {
      a0 = S0[frow * kDv + 16 * cq + 2 * m];
      a1 = S0[frow * kDv + 16 * cq + 2 * m + 1];
    }
    W[m] = pk2(a0, a1);
  }
  if (!kKeys && z0 && cq == 3) w64 = z0[frow];

  // chain-rule thread map (tid < 128): token ct, dimension ca of the group
  const int ct = tid >> 3, ca = grp * 8 + (tid & 7);
  const float om = omega[h * kD + ca], ph = phi[h * kD + ca];
  float acc_g = 0.f, acc_o = 0.f, acc_p = 0.f;
  const Tin* vsrc = kKeys ? q : k;     // tensor whose features are the values
  const Tin* usrc = kKeys ? k : q;     // tensor whose gradient this pass writes

  for (int c0 = 0; c0 < T; c0 += kFsaCT) {
    const int nc = min(kFsaCT, T - c0);
    __syncthreads();   // the previous chunk is done with every buffer
    for (int e = tid; e < kFsaCT * kQP; e += blockDim.x) {
      const int t = e / kQP, col = e % kQP;
      float gq = 0.f, vv = 0.f;
      if (t < nc && col <= kDv) {
        const int64_t r = seq + row(c0 + t);
        gq = col < kDv ? dN[r * kDv + col] : dD[r];
        vv = col < kDv ? load_as_float(v + r * kDv + col) : 1.0f;
      }
      sm.qa[t][col] = kKeys ? vv : gq;
      sm.kb[t][col] = kKeys ? gq : vv;
    }
    if (tid < 128) {
      float* dst = &sm.pv[ct][kCh * (tid & 7)];
      if (ct < nc) {
        const int r = row(c0 + ct);
        float ch[kCh];
        harmonic_channels<N>(load_as_float(vsrc + (seq + r) * kD + ca), g, om,
                             phase_mod_2pi(pos0 + r, ph), ch);
#pragma unroll
        for (int cc = 0; cc < kCh; ++cc) dst[cc] = ch[cc];
      } else {
#pragma unroll
        for (int cc = 0; cc < kCh; ++cc) dst[cc] = 0.f;
      }
    }
    __syncthreads();
    if (tid < kFsaCT * kFsaCT) {
      const int t = tid >> 4, j = tid & (kFsaCT - 1);
      if (j <= t) {
        const ulonglong2* a = reinterpret_cast<const ulonglong2*>(&sm.qa[t][0]);
        const ulonglong2* b = reinterpret_cast<const ulonglong2*>(&sm.kb[j][0]);
        uint64_t s0 = 0, s1 = 0;
#pragma unroll
        for (int i = 0; i < kQP / 4; ++i) {
          const ulonglong2 x = a[i], y = b[i];
          s0 = ffma2(x.x, y.x, s0);
          s1 = ffma2(x.y, y.y, s1);
        }
        float p0, p1, p2, p3;
        upk2(s0, p0, p1);
        upk2(s1, p2, p3);
        sm.ds[t][j] = (p0 + p1) + (p2 + p3);
      }
    }
    // state readout of the chunk per column quarter (before this chunk's keys)
#pragma unroll 2
    for (int t = 0; t < kFsaCT; ++t) {
      const ulonglong2* a = reinterpret_cast<const ulonglong2*>(&sm.qa[t][16 * cq]);
      uint64_t acc2 = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const ulonglong2 x = a[i];
        acc2 = ffma2(x.x, W[2 * i], acc2);
        acc2 = ffma2(x.y, W[2 * i + 1], acc2);
      }
      float x0, x1;
      upk2(acc2, x0, x1);
      float acc = x0 + x1;
      if (cq == 3) acc = fmaf(sm.qa[t][kDv], w64, acc);
      sm.part[cq][t][f] = acc;
    }
    __syncthreads();
    // feature gradients: the four quarters plus the intra-chunk pairs, tokens
    // cq, cq + 4, cq + 8, cq + 12 of row f
#pragma unroll
    for (int m = 0; m < kFsaCT / 4; ++m) {
      const int t = cq + 4 * m;
      float acc = (sm.part[0][t][f] + sm.part[1][t][f]) + (sm.part[2][t][f] + sm.part[3][t][f]);
      for (int j = 0; j <= t; ++j) acc = fmaf(sm.ds[t][j], sm.pv[j][f], acc);
      sm.part[0][t][f] = acc;
    }
    __syncthreads();
    // state update W += pv^T kb (pv and kb are zero past the end)
#pragma unroll 4
    for (int j = 0; j < kFsaCT; ++j) {
      const float w = sm.pv[j][f];
      const uint64_t w2 = pk2(w, w);
      const ulonglong2* b = reinterpret_cast<const ulonglong2*>(&sm.kb[j][16 * cq]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const ulonglong2 x = b[i];
        W[2 * i] = ffma2(x.x, w2, W[2 * i]);
        W[2 * i + 1] = ffma2(x.y, w2, W[2 * i + 1]);
      }
      if (cq == 3) w64 = fmaf(w, sm.kb[j][kDv], w64);
    }
    // chain rule of the chunk's tokens for the group's dimensions
    if (tid < 128 && ct < nc) {
      const int r = row(c0 + ct);
      const int64_t pos = pos0 + r;
      const HarmGrad e = harmonic_vjp<N>(load_as_float(usrc + (seq + r) * kD + ca), g, om,
                                         phase_mod_2pi(pos, ph), static_cast<float>(pos),
                                         &sm.part[0][ct][kCh * (tid & 7)]);
      dout[(seq + r) * kD + ca] = store_from_float<Tin>(e.du);
      acc_g += e.dgamma;
      acc_o += e.domega;
      acc_p += e.dphi;
    }
  }
  // parameter gradients: sum over the 16 tokens of each dimension, then atomics
  if (tid < 128) {
#pragma unroll
    for (int off = 8; off < 32; off <<= 1) {
      acc_g += __shfl_xor_sync(0xffffffffu, acc_g, off);
      acc_o += __shfl_xor_sync(0xffffffffu, acc_o, off);
      acc_p += __shfl_xor_sync(0xffffffffu, acc_p, off);
    }
    if ((tid & 31) < 8) {
      sm.red[tid >> 5][tid & 7][0] = acc_g;
      sm.red[tid >> 5][tid & 7][1] = acc_o;
      sm.red[tid >> 5][tid & 7][2] = acc_p;
    }
  }
  __syncthreads();
  if (tid < 8) {
    float sg = 0.f, so = 0.f, sp = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      sg += sm.red[w][tid][0];
      so += sm.red[w][tid][1];
      sp += sm.red[w][tid][2];
    }
    atomicAdd(&domega[h * kD + grp * 8 + tid], so);
    if (dphi) atomicAdd(&dphi[h * kD + grp * 8 + tid], sp);
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) sg += __shfl_xor_sync(0xffu, sg, off);
    if (tid == 0) atomicAdd(&dgamma[h], sg);
  }
}

// resident CTAs per SM the register budget is set for (320 threads at N = 2,
// 448 at N = 3)
template <int N>
constexpr int fsa_min_blocks() { return N == 2 ? 3 : 2; }

template <int N, typename Tin>
__global__ void __launch_bounds__(4 * 8 * Harm<N>::kCh, fsa_min_blocks<N>()) fsa_harmonic_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
    const float* __restrict__ dN, const float* __restrict__ dD, const float* __restrict__ gamma,
    const float* __restrict__ omega, const float* __restrict__ phi, int H, int T, int64_t pos0,
    const float* __restrict__ S0, const float* __restrict__ z0, Tin* __restrict__ dq,
    Tin* __restrict__ dk, float* __restrict__ dgamma, float* __restrict__ domega,
    float* __restrict__ dphi) {
  __shared__ FsaSmem<N> sm;
  if (blockIdx.y == 0)
    fsa_pass<N, Tin, false>(q, k, v, dN, dD, gamma, omega, phi, H, T, pos0, S0, z0, dq, dgamma,
                            domega, dphi, sm);
  else
    fsa_pass<N, Tin, true>(q, k, v, dN, dD, gamma, omega, phi, H, T, pos0, S0, z0, dk, dgamma,
                           domega, dphi, sm);
}

template <int N, typename Tin, typename Tg>
cudaError_t bwd_h(const ChunkBwdArgs& a, cudaStream_t st) {
  const ChunkFwdArgs& f = a.f;
  const int64_t rows = static_cast<int64_t>(f.B) * f.H * f.T;
  float* dN = static_cast<float*>(a.workspace);
  float* dD = dN + rows * kDv;
  cudaError_t e;
  if ((e = cudaMemsetAsync(a.dgamma, 0, sizeof(float) * f.H, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(a.domega, 0, sizeof(float) * f.H * kD, st)) != cudaSuccess) return e;
  if (a.dphi && (e = cudaMemsetAsync(a.dphi, 0, sizeof(float) * f.H * kD, st)) != cudaSuccess)
    return e;
  if (rows == 0) return cudaSuccess;
  harm_bwd_prep_kernel<Tg>
      <<<static_cast<unsigned>((rows + kPrepRows - 1) / kPrepRows), 32 * kPrepRows, 0, st>>>(
      a.o, a.Dn, static_cast<const Tg*>(a.dO), f.eps, rows, dN, dD);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // dv: the forward recurrence in reverse time with queries k, keys q, values dN
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(f.B * f.H) * kRanks);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kRanks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, chunk_fwd_harmonic_kernel<N, Tin, float, Tin, true>,
                         static_cast<const Tin*>(f.k), static_cast<const Tin*>(f.q),
                         static_cast<const float*>(dN), f.gamma, f.omega, f.phi, f.H, f.T,
                         f.pos0, 0.0f, static_cast<const float*>(nullptr),
                         static_cast<const float*>(nullptr), static_cast<Tin*>(a.dv),
                         static_cast<float*>(nullptr), static_cast<float*>(nullptr),
                         static_cast<float*>(nullptr));
  if (e != cudaSuccess) return e;
  // dq and dk: the two feature-space passes in one launch
  const dim3 grid(static_cast<unsigned>(f.B * f.H) * 8, 2);
  fsa_harmonic_kernel<N, Tin><<<grid, 4 * 8 * Harm<N>::kCh, 0, st>>>(
      static_cast<const Tin*>(f.q), static_cast<const Tin*>(f.k), static_cast<const Tin*>(f.v), dN,
      dD, f.gamma, f.omega, f.phi, f.H, f.T, f.pos0, f.S0, f.z0, static_cast<Tin*>(a.dq),
      static_cast<Tin*>(a.dk), a.dgamma, a.domega, a.dphi);
  return cudaGetLastError();
}

template <int N>
cudaError_t bwd_n(const ChunkBwdArgs& a, cudaStream_t st) {
  const bool in_f32 = a.f.in_dtype == SANATAN_F32;
  const bool g_f32 = a.grad_dtype == SANATAN_F32;
  if (in_f32 && g_f32) return bwd_h<N, float, float>(a, st);
  if (in_f32) return bwd_h<N, float, __nv_bfloat16>(a, st);
  if (g_f32) return bwd_h<N, __nv_bfloat16, float>(a, st);
  return bwd_h<N, __nv_bfloat16, __nv_bfloat16>(a, st);
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

template <int N, typename Tin>
cudaError_t chunk_h(const ChunkFwdArgs& a, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B * a.H) * kRanks);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kRanks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chunk_fwd_harmonic_kernel<N, Tin, Tin, float, false>,
                            static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k),
                            static_cast<const Tin*>(a.v), a.gamma, a.omega, a.phi, a.H, a.T,
                            a.pos0, a.eps, a.S0, a.z0, a.o, a.D, a.S_out, a.z_out);
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
  if (harmonics == 2) return f32 ? chunk_h<2, float>(a, st) : chunk_h<2, __nv_bfloat16>(a, st);
  if (harmonics == 3) return f32 ? chunk_h<3, float>(a, st) : chunk_h<3, __nv_bfloat16>(a, st);
  return cudaErrorInvalidValue;
}

size_t chunk_bwd_harmonic_workspace_bytes(int B, int H, int T, int harmonics) {
  if (harmonics < 2) return 0;
  return static_cast<size_t>(B) * H * T * (kDv + 1) * sizeof(float);
}

cudaError_t chunk_bwd_harmonic_launch(const ChunkBwdArgs& a, int harmonics, cudaStream_t st) {
  if (harmonics == 1) return chunk_bwd_simt_launch(a, st);
  if (harmonics == 2) return bwd_n<2>(a, st);
  if (harmonics == 3) return bwd_n<3>(a, st);
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
