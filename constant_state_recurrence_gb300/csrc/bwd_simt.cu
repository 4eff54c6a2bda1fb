// Backward of the chunked p=1 attention on the CUDA cores, all in float32.
//
// The pages give no gradient; this is the chain rule through the feature
// map (reading notes §2.2-§2.3, eqs. (2)-(6)) and the normalised causal sum
// of eq. (9).  With N_t = sum_{j<=t} s_tj v_j (+ Phi(q_t) S0),
// D_t = sum_{j<=t} s_tj (+ Phi(q_t) z0) and o_t = N_t / (D_t + eps):
//   dN_t  = dO_t / (D_t + eps),        dD_t = -(dO_t . o_t) / (D_t + eps)
//   ds_tj = [j <= t] (dN_t . v_j + dD_t)
//   dPhi(q_t) = sum_j ds_tj Phi(k_j) + S_{t-} dN_t + z_{t-} dD_t   (S_{t-}: state before the chunk)
//   dPhi(k_j) = sum_t ds_tj Phi(q_t) + G v_j + g                   (G, g: sums over later chunks)
//   dv_j      = sum_t [j <= t] s_tj dN_t + G^T Phi(k_j)
// with G = sum_{later t} Phi(q_t) dN_t^T and g = sum_{later t} Phi(q_t) dD_t.
// One CTA per (batch, head): a forward sweep over the chunks carries S, z and
// produces dq; a reverse sweep carries G, g and produces dk, dv.  Parameter
// gradients (gamma, omega, phi) are reduced per CTA and added atomically.
#include "sanatan_internal.h"
#include "sanatan_math.cuh"

namespace sanatan {
namespace {

constexpr int kD = 64;
constexpr int kDv = 64;
constexpr int kF = 6 * kD;
constexpr int kFP = kF + 1;   // padded feature stride
constexpr int kC = 32;
constexpr int kVP = kDv + 1;  // padded value stride
constexpr int kThreads = 256;

struct BwdSmem {
  float pq[kC * kFP];     // Phi(Q) of the chunk (reverse sweep)
  float pk[kC * kFP];     // Phi(K) of the chunk
  float v[kC * kVP];
  float dn[kC * kVP];
  float dd[kC];
  float st[kF * kDv];     // S (forward sweep) or G (reverse sweep)
  float sz[kF];           // z or g
  float P[kC * (kC + 1)];
  float dS[kC * (kC + 1)];
  float red[kThreads / 32][2 * kD + 1];
};

// Everything of one (token, dim) element that the chain rule needs.
struct ElemGrad {
  float du, dgamma, domega, dphi;
};

__device__ __forceinline__ ElemGrad feature_vjp(float u, float g, float om, float phase, float t,
                                                const float (&dphi)[6]) {
  const float th = squash_exact(u);
  float sx, cx;
  sincosf(th + om, &sx, &cx);
  const float gx = cx - sx;
  const float gpx = -sx - cx;
  const float r = tanhf(g * gx);
  float sr, cr;
  sincosf(th + phase, &sr, &cr);
  const float dc = dphi[1] + r * dphi[4];
  const float ds = dphi[2] + r * dphi[5];
  const float dr = dphi[3] + cr * dphi[4] + sr * dphi[5];
  const float dth_rot = -sr * dc + cr * ds;
  const float dpre = dr * (1.0f - r * r);
  const float dtheta = dth_rot + dpre * g * gpx;
  const float den = 1.0f + fabsf(u);
  ElemGrad e;
  e.du = dtheta * kPi / (den * den);
  e.dgamma = dpre * gx;
  e.domega = dpre * g * gpx;
  e.dphi = dth_rot * t;
  return e;
}

template <typename Tin>
__device__ __forceinline__ void load_features(const Tin* __restrict__ src, int64_t row0, int nc,
                                              int h, const float* __restrict__ omega,
                                              const float* __restrict__ phi, float g,
                                              int64_t pos, float* dst, int tid) {
  for (int e = tid; e < kC * kD; e += kThreads) {
    const int t = e / kD, a = e % kD;
    float* out = dst + t * kFP + 6 * a;
    if (t < nc) {
      const float u = load_as_float(src + (row0 + t) * kD + a);
      const FeatAngles f =
          feat_exact(u, g, omega[h * kD + a], phase_mod_2pi(pos + t, phi[h * kD + a]));
      float ch[6];
      feat_channels(f, ch);
#pragma unroll
      for (int c = 0; c < 6; ++c) out[c] = ch[c];
    } else {
#pragma unroll
      for (int c = 0; c < 6; ++c) out[c] = 0.f;
    }
  }
}

// dN, dD and v of a chunk.
template <typename Tin, typename Tg>
__device__ __forceinline__ void load_grads(const Tin* __restrict__ v, const Tg* __restrict__ dO,
                                           const float* __restrict__ o,
                                           const float* __restrict__ Dn, float eps, int64_t row0,
                                           int nc, BwdSmem& sm, int tid, int warp, int lane) {
  for (int e = tid; e < kC * kDv; e += kThreads) {
    const int t = e / kDv, c = e % kDv;
    float vv = 0.f, dn = 0.f;
    if (t < nc) {
      vv = load_as_float(v + (row0 + t) * kDv + c);
      dn = load_as_float(dO + (row0 + t) * kDv + c) / (Dn[row0 + t] + eps);
    }
    sm.v[t * kVP + c] = vv;
    sm.dn[t * kVP + c] = dn;
  }
  // dD_t = -(dO_t . o_t) / (D_t + eps): one warp per 4 tokens
  for (int t = warp; t < kC; t += kThreads / 32) {
    float acc = 0.f;
    if (t < nc) {
      for (int c = lane; c < kDv; c += 32)
        acc += load_as_float(dO + (row0 + t) * kDv + c) * o[(row0 + t) * kDv + c];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) sm.dd[t] = (t < nc) ? -acc / (Dn[row0 + t] + eps) : 0.f;
  }
}

template <typename Tin, typename Tg>
__global__ void __launch_bounds__(kThreads, 1) chunk_bwd_simt_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
    const float* __restrict__ gamma, const float* __restrict__ omega,
    const float* __restrict__ phi, int H, int T, int64_t pos0, float eps,
    const float* __restrict__ S0, const float* __restrict__ z0, const float* __restrict__ o,
    const float* __restrict__ Dn, const Tg* __restrict__ dO, Tin* __restrict__ dq,
    Tin* __restrict__ dk, Tin* __restrict__ dv, float* __restrict__ dgamma,
    float* __restrict__ domega, float* __restrict__ dphi) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
  const int bh = blockIdx.x;
  const int h = bh % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t seq = static_cast<int64_t>(bh) * T;
  const float g = gamma[h];
  // The element tasks of a thread: dimension a, tokens tb + 4i.
  const int a = tid % kD;
  const int tb = tid / kD;
  const float om = omega[h * kD + a];
  const float ph = phi[h * kD + a];
  float acc_g = 0.f, acc_om = 0.f, acc_ph = 0.f;

  // ---------------------------------------------------------------- forward sweep: dq
  for (int i = tid; i < kF * kDv; i += kThreads)
    sm.st[i] = S0 ? S0[static_cast<int64_t>(bh) * kF * kDv + i] : 0.f;
  for (int i = tid; i < kF; i += kThreads) sm.sz[i] = z0 ? z0[static_cast<int64_t>(bh) * kF + i] : 0.f;
  for (int c0 = 0; c0 < T; c0 += kC) {
    const int nc = min(kC, T - c0);
    __syncthreads();
    load_features(k, seq + c0, nc, h, omega, phi, g, pos0 + c0, sm.pk, tid);
    load_grads(v, dO, o, Dn, eps, seq + c0, nc, sm, tid, warp, lane);
    __syncthreads();
    // dS[t][j] = [j <= t] (dN_t . v_j + dD_t)
    {
      const int t = tid >> 3;
#pragma unroll
      for (int m = 0; m < kC / 8; ++m) {
        const int j = (tid & 7) + 8 * m;
        float s = 0.f;
        if (j <= t) {
          for (int e = 0; e < kDv; ++e) s = fmaf(sm.dn[t * kVP + e], sm.v[j * kVP + e], s);
          s += sm.dd[t];
        }
        sm.dS[t * (kC + 1) + j] = s;
      }
    }
    __syncthreads();
    // dPhi(q_t) for the six channels of dim a, then the chain rule.
    for (int t = tb; t < nc; t += kThreads / kD) {
      float dphi6[6];
#pragma unroll
      for (int c = 0; c < 6; ++c) {
        const int f = 6 * a + c;
        float s = 0.f;
        for (int j = 0; j <= t; ++j) s = fmaf(sm.dS[t * (kC + 1) + j], sm.pk[j * kFP + f], s);
        for (int e0 = 0; e0 < kDv; ++e0) {
          const int e = (e0 + lane) & (kDv - 1);
          s = fmaf(sm.st[f * kDv + e], sm.dn[t * kVP + e], s);
        }
        dphi6[c] = fmaf(sm.sz[f], sm.dd[t], s);
      }
      const int64_t tabs = pos0 + c0 + t;
      const ElemGrad eg = feature_vjp(load_as_float(q + (seq + c0 + t) * kD + a), g, om,
                                      phase_mod_2pi(tabs, ph), static_cast<float>(tabs), dphi6);
      dq[(seq + c0 + t) * kD + a] = store_from_float<Tin>(eg.du);
      acc_g += eg.dgamma;
      acc_om += eg.domega;
      acc_ph += eg.dphi;
    }
    __syncthreads();
    // S += Phi(K)^T V, z += column sums of Phi(K)
    {
      const int e = tid & (kDv - 1);
      for (int f = tid >> 6; f < kF; f += kThreads / kDv) {
        float s = sm.st[f * kDv + e];
        for (int j = 0; j < nc; ++j) s = fmaf(sm.pk[j * kFP + f], sm.v[j * kVP + e], s);
        sm.st[f * kDv + e] = s;
      }
      for (int f = tid; f < kF; f += kThreads) {
        float s = sm.sz[f];
        for (int j = 0; j < nc; ++j) s += sm.pk[j * kFP + f];
        sm.sz[f] = s;
      }
    }
  }

  // ---------------------------------------------------------------- reverse sweep: dk, dv
  __syncthreads();
  for (int i = tid; i < kF * kDv; i += kThreads) sm.st[i] = 0.f;
  for (int i = tid; i < kF; i += kThreads) sm.sz[i] = 0.f;
  const int nchunks = (T + kC - 1) / kC;
  for (int ci = nchunks - 1; ci >= 0; --ci) {
    const int c0 = ci * kC;
    const int nc = min(kC, T - c0);
    __syncthreads();
    load_features(q, seq + c0, nc, h, omega, phi, g, pos0 + c0, sm.pq, tid);
    load_features(k, seq + c0, nc, h, omega, phi, g, pos0 + c0, sm.pk, tid);
    load_grads(v, dO, o, Dn, eps, seq + c0, nc, sm, tid, warp, lane);
    __syncthreads();
    // P[t][j] and dS[t][j], both masked to j <= t.
    {
      const int t = tid >> 3;
#pragma unroll
      for (int m = 0; m < kC / 8; ++m) {
        const int j = (tid & 7) + 8 * m;
        float p = 0.f, s = 0.f;
        if (j <= t) {
          for (int f = 0; f < kF; ++f) p = fmaf(sm.pq[t * kFP + f], sm.pk[j * kFP + f], p);
          for (int e = 0; e < kDv; ++e) s = fmaf(sm.dn[t * kVP + e], sm.v[j * kVP + e], s);
          s += sm.dd[t];
        }
        sm.P[t * (kC + 1) + j] = p;
        sm.dS[t * (kC + 1) + j] = s;
      }
    }
    __syncthreads();
    // dPhi(k_j) and the chain rule for k.
    for (int j = tb; j < nc; j += kThreads / kD) {
      float dphi6[6];
#pragma unroll
      for (int c = 0; c < 6; ++c) {
        const int f = 6 * a + c;
        float s = 0.f;
        for (int t = j; t < kC; ++t) s = fmaf(sm.dS[t * (kC + 1) + j], sm.pq[t * kFP + f], s);
        for (int e0 = 0; e0 < kDv; ++e0) {
          const int e = (e0 + lane) & (kDv - 1);
          s = fmaf(sm.st[f * kDv + e], sm.v[j * kVP + e], s);
        }
        dphi6[c] = s + sm.sz[f];
      }
      const int64_t tabs = pos0 + c0 + j;
      const ElemGrad eg = feature_vjp(load_as_float(k + (seq + c0 + j) * kD + a), g, om,
                                      phase_mod_2pi(tabs, ph), static_cast<float>(tabs), dphi6);
      dk[(seq + c0 + j) * kD + a] = store_from_float<Tin>(eg.du);
      acc_g += eg.dgamma;
      acc_om += eg.domega;
      acc_ph += eg.dphi;
    }
    // dv_j = sum_{t >= j} P[t][j] dN_t + G^T Phi(k_j)
    {
      const int e = tid & (kDv - 1);
      for (int j = tid >> 6; j < nc; j += kThreads / kDv) {
        float s = 0.f;
        for (int t = j; t < kC; ++t) s = fmaf(sm.P[t * (kC + 1) + j], sm.dn[t * kVP + e], s);
        for (int f = 0; f < kF; ++f) s = fmaf(sm.pk[j * kFP + f], sm.st[f * kDv + e], s);
        dv[(seq + c0 + j) * kDv + e] = store_from_float<Tin>(s);
      }
    }
    __syncthreads();
    // G += Phi(Q)^T dN, g += Phi(Q)^T dD
    {
      const int e = tid & (kDv - 1);
      for (int f = tid >> 6; f < kF; f += kThreads / kDv) {
        float s = sm.st[f * kDv + e];
        for (int t = 0; t < nc; ++t) s = fmaf(sm.pq[t * kFP + f], sm.dn[t * kVP + e], s);
        sm.st[f * kDv + e] = s;
      }
      for (int f = tid; f < kF; f += kThreads) {
        float s = sm.sz[f];
        for (int t = 0; t < nc; ++t) s = fmaf(sm.pq[t * kFP + f], sm.dd[t], s);
        sm.sz[f] = s;
      }
    }
  }

  // ---------------------------------------------------------------- parameter gradients
  // Threads tid and tid + 64k share dimension a: reduce through shared memory.
  __syncthreads();
  float* red = &sm.red[0][0];  // [4 token lanes][2*64 + 1] reused as scratch
  if (tid < kThreads) {
    red[(tid / kD) * (2 * kD + 1) + a] = acc_om;
    red[(tid / kD) * (2 * kD + 1) + kD + a] = acc_ph;
  }
  float gsum = acc_g;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) gsum += __shfl_xor_sync(0xffffffffu, gsum, off);
  __shared__ float s_g[kThreads / 32];
  if (lane == 0) s_g[warp] = gsum;
  __syncthreads();
  if (tid < kD) {
    float so = 0.f, sp = 0.f;
    for (int r = 0; r < kThreads / kD; ++r) {
      so += red[r * (2 * kD + 1) + tid];
      sp += red[r * (2 * kD + 1) + kD + tid];
    }
    atomicAdd(&domega[h * kD + tid], so);
    if (dphi) atomicAdd(&dphi[h * kD + tid], sp);
  }
  if (tid == 0) {
    float s = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) s += s_g[w];
    atomicAdd(&dgamma[h], s);
  }
}

template <typename Tin, typename Tg>
cudaError_t launch(const ChunkBwdArgs& a, cudaStream_t st) {
  const ChunkFwdArgs& f = a.f;
  const size_t smem = sizeof(BwdSmem);
  auto kern = chunk_bwd_simt_kernel<Tin, Tg>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(a.dgamma, 0, sizeof(float) * f.H, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(a.domega, 0, sizeof(float) * f.H * kD, st)) != cudaSuccess) return e;
  if (a.dphi && (e = cudaMemsetAsync(a.dphi, 0, sizeof(float) * f.H * kD, st)) != cudaSuccess)
    return e;
  if (f.B * f.H == 0) return cudaSuccess;
  const ProfileEvents& pe = profile_events();
  if (pe.start != nullptr) cudaEventRecord(pe.start, st);
  kern<<<f.B * f.H, kThreads, smem, st>>>(
      static_cast<const Tin*>(f.q), static_cast<const Tin*>(f.k), static_cast<const Tin*>(f.v),
      f.gamma, f.omega, f.phi, f.H, f.T, f.pos0, f.eps, f.S0, f.z0, a.o, a.Dn,
      static_cast<const Tg*>(a.dO), static_cast<Tin*>(a.dq), static_cast<Tin*>(a.dk),
      static_cast<Tin*>(a.dv), a.dgamma, a.domega, a.dphi);
  e = cudaGetLastError();
  if (pe.stop != nullptr) cudaEventRecord(pe.stop, st);
  return e;
}

}  // namespace

size_t chunk_bwd_simt_smem_bytes() { return sizeof(BwdSmem); }

cudaError_t chunk_bwd_simt_launch(const ChunkBwdArgs& a, cudaStream_t st) {
  const bool in_f32 = a.f.in_dtype == SANATAN_F32;
  const bool g_f32 = a.grad_dtype == SANATAN_F32;
  if (in_f32 && g_f32) return launch<float, float>(a, st);
  if (in_f32) return launch<float, __nv_bfloat16>(a, st);
  if (g_f32) return launch<__nv_bfloat16, float>(a, st);
  return launch<__nv_bfloat16, __nv_bfloat16>(a, st);
}

}  // namespace sanatan
