// Gradients of the power-sharpened causal attention (eq. (8) of "SANATAN:
// Root-Parity Gated Angular Attention with an Exact Constant-State Recurrent
// Form", reading notes §2.6) on the tensor cores.  The pages give no
// gradient; with x_tj = s_tj / 4d, w_tj = [j <= t] x_tj^p, D_t = sum_j w_tj,
// Dh_t = D_t + eps and o_t = sum_j w_tj v_j / Dh_t, the chain rule gives
//   dN_t = dO_t / Dh_t,   dD_t = -(dO_t . o_t) / Dh_t,
//   ds_tj = [j <= t] (dN_t . v_j + dD_t) p x_tj^(p-1) / 4d,
//   dv_j = sum_t w_tj dN_t,
//   dPhi(q_t) = sum_j ds_tj Phi(k_j),   dPhi(k_j) = sum_t ds_tj Phi(q_t),
// and then the feature map's own chain rule (eqs. (2)-(4), (6)) to dq, dk and
// the per-head dgamma, domega, dphi.
//
// Launches: the forward's preparation kernel (Phi(Q), Phi(K), [V | 1 | 0]
// per chunk), a small kernel for dN (bf16, operand layout) and dD, then two
// tensor-core passes, each one CTA per (sequence, chunk) with all 320 features:
//   query pass: per query chunk i, for the 64-key halves of the key chunks
//     j <= i: S = Phi(Q_i) Phi(K_j,half)^T, dW = dN_i V_j,half^T, the epilogue
//     forms dS in its own TMEM buffer while the next half's S and dW are
//     computed, and dPhi(Q_i) += dS Phi(K_j,half);
//   key pass: per key chunk j, for the 64-query halves of the query chunks
//     i >= j: S^T, dW^T likewise, the weights W^T and dS^T in place, then
//     dPhi(K_j) += dS^T Phi(Q_i,half) and dv_j += W^T dN_i,half.
// Halves of 64 tokens keep scores, score gradients and the 320-column feature
// gradient inside the 512 TMEM columns without splitting the features, so
// every score is computed once per pass; the streamed halves are
// double-buffered in shared memory.  After its last tile each CTA applies the
// feature map's chain rule and writes du, and adds its share of dgamma,
// domega, dphi with atomics.
#include "pow_common.cuh"
#include "sanatan_internal.h"
#include "sanatan_math.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace sanatan {

__device__ int g_pow_bwd_error;  // set when a bounded wait gives up

namespace {

using namespace tc;
using namespace tcc;
using namespace powc;

constexpr uint32_t kDNBytes = 16 * 1024;   // dN of one chunk: [tg * 1024 + ng * 128 + r * 16]
constexpr uint32_t kDDBytes = kC * 4;      // dD of one chunk (f32)

// TMEM columns (every access stays inside the 512 allocated).  Query pass:
constexpr uint32_t kQTF = 0;      // dPhi(Q_i), 320 columns
constexpr uint32_t kQTS = 320;    // scores of a 64-key half (f32)
constexpr uint32_t kQTDW = 384;   // dW of the half (f32)
constexpr uint32_t kQTDS = 448;   // dS of the half: bf16 hi | lo per 32-key block
// Key pass:
constexpr uint32_t kKTS = 0;      // S^T of a 64-query half, then W^T hi | lo in place
constexpr uint32_t kKTDW = 64;    // dW^T, then dS^T hi | lo in place
constexpr uint32_t kKTF = 128;    // dPhi(K_j), 320 columns
constexpr uint32_t kKTV = 448;    // dv_j, 64 columns
constexpr uint32_t kTmemCols = 512;

// Bytes of one 64-token half of a chunk's operands.
constexpr uint32_t kHalfPhi = 8 * kXQ;      // Phi: eight token groups
constexpr uint32_t kHalfV = 8 * kVGroup;    // [V | 1 | 0]
constexpr uint32_t kHalfDN = 8 * 1024;      // dN
constexpr uint32_t kHalfDD = 64 * 4;        // dD

enum Bar {
  kResFull = 0, kStrFull0, kStrFull1, kSDone, kSFree, kDSReady, kTileDone0, kTileDone1, kDrain,
  kNumBars
};

constexpr int kEpiWarps = 8;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kThreads = 32 * (kLoadWarp + 1);
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kSeqGroup = 8;    // CTAs run in groups of this many sequences (L2 reuse)

struct Misc {
  uint64_t bar[kNumBars];
  uint32_t tmem_base;
  int abort_flag;
  float red_omega[64];   // this CTA's share of domega, dphi and dgamma
  float red_phi[64];
  float red_gamma;
};

struct BwdParams {
  const unsigned char* ws;    // per (sequence, chunk): Phi(Q) | Phi(K) | [V | 1 | 0]
  const unsigned char* dn;    // per (sequence, chunk): dN, kDNBytes
  const float* dd;            // per (sequence, chunk): dD, 128 floats
  const __nv_bfloat16* u;     // raw q (query pass) or k (key pass) [B, H, T, 64]
  const float* gamma;
  const float* omega;
  const float* phi;
  int H, T, nchunks, bhn;
  int64_t pos0;
  int64_t pos_mid;            // pos0 + (T - 1) / 2: the reference position of the phi gradient
  __nv_bfloat16* du;          // dq or dk
  __nv_bfloat16* dv;          // key pass only
  float* dgamma;
  float* domega;
  float* dphi;                // may be null
};

struct DPrepParams {
  const void* dO;
  int grad_bf16;
  const float* o;
  const float* D;
  float eps;
  int T, nchunks;
  int64_t ntok;               // bhn * nchunks * 128
  unsigned char* dn;
  float* dd;
};

__device__ __forceinline__ bool wait_bar(Misc& m, int b, uint32_t parity) {
  if (*reinterpret_cast<volatile int*>(&m.abort_flag)) return false;
  if (mbar_wait_bounded(&m.bar[b], parity, kWaitNs)) return true;
  m.abort_flag = 1;
  atomicOr(&g_pow_bwd_error, 1);
  return false;
}

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
}

// ---------------------------------------------------------------------------
// dN = dO / Dh (bf16, the operand layout of a chunk) and dD = -(dO . o) / Dh,
// zero for the padding rows of the last chunk.  Eight threads per token, eight
// columns each.
__global__ void __launch_bounds__(256) pow_dprep_kernel(DPrepParams prm) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t tok = g >> 3;          // (sequence, chunk, row), row fastest
  const int ng = static_cast<int>(g & 7);
  const bool in_range = tok < prm.ntok;
  const int row = static_cast<int>(tok % kC);
  const int64_t sc = tok / kC;         // sequence * nchunks + chunk
  const int chunk = static_cast<int>(sc % prm.nchunks);
  const int64_t bh = sc / prm.nchunks;
  const int t = chunk * kC + row;
  const bool valid = in_range && t < prm.T;
  float dov[8], ov[8];
  float dh = 1.0f;
  if (valid) {
    const int64_t grow = bh * prm.T + t;
    if (prm.grad_bf16) {
      const uint4 w = ldg_nc_v4(static_cast<const __nv_bfloat16*>(prm.dO) + grow * kD + 8 * ng);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        dov[2 * i] = __uint_as_float(ww[i] << 16);
        dov[2 * i + 1] = __uint_as_float(ww[i] & 0xffff0000u);
      }
    } else {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(prm.dO) +
                                                        grow * kD + 8 * ng);
      const float4 a = p[0], b = p[1];
      dov[0] = a.x; dov[1] = a.y; dov[2] = a.z; dov[3] = a.w;
      dov[4] = b.x; dov[5] = b.y; dov[6] = b.z; dov[7] = b.w;
    }
    const float4* po = reinterpret_cast<const float4*>(prm.o + grow * kD + 8 * ng);
    const float4 a = po[0], b = po[1];
    ov[0] = a.x; ov[1] = a.y; ov[2] = a.z; ov[3] = a.w;
    ov[4] = b.x; ov[5] = b.y; ov[6] = b.z; ov[7] = b.w;
    dh = prm.D[grow] + prm.eps;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) { dov[i] = 0.f; ov[i] = 0.f; }
  }
  const float inv = 1.0f / dh;
  float dot = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) dot = fmaf(dov[i], ov[i], dot);
  dot += __shfl_xor_sync(0xffffffffu, dot, 1);
  dot += __shfl_xor_sync(0xffffffffu, dot, 2);
  dot += __shfl_xor_sync(0xffffffffu, dot, 4);
  if (!in_range) return;
  uint4 packed;
  packed.x = pack_bf16x2(dov[0] * inv, dov[1] * inv);
  packed.y = pack_bf16x2(dov[2] * inv, dov[3] * inv);
  packed.z = pack_bf16x2(dov[4] * inv, dov[5] * inv);
  packed.w = pack_bf16x2(dov[6] * inv, dov[7] * inv);
  unsigned char* dst = prm.dn + sc * static_cast<int64_t>(kDNBytes) + (row >> 3) * 1024 + ng * 128 +
                       (row & 7) * 16;
  *reinterpret_cast<uint4*>(dst) = packed;
  if (ng == 0) prm.dd[sc * kC + row] = valid ? -dot * inv : 0.f;
}

// ---------------------------------------------------------------------------
// The feature map's chain rule for one token and the 16 dimensions
// 32 fh + 16 ch .. + 15 (two groups of eight), reading the feature gradients of
// this CTA's half from TMEM: inside the half, dimension group ag' (0..3) holds
// channels c = 1..5 in columns 40 ag' + 8 (c - 1) + e for dimension 8 ag' + e.
//   dc = d1 + r d4, ds = d2 + r d5, dr = d3 + c d4 + s d5,
//   dth_rot = -s dc + c ds, dpre = dr (1 - r^2),
//   dtheta = dth_rot + dpre gamma g'(theta + omega), du = dtheta pi / (1 + |u|)^2,
//   dgamma += dpre g, domega += dpre gamma g', dphi += dth_rot (t - t_mid),
// with g(x) = cos x - sin x, g'(x) = -sin x - cos x.  The outputs do not
// change when every position of a sequence moves by the same amount (each
// score depends on positions only through t - j), so for every dimension the
// phase gradients dth_rot of all q and k tokens of a sequence sum to zero and
// sum_t dth_rot t = sum_t dth_rot (t - t_mid) exactly; the second form, with
// t_mid the middle position, keeps a large position offset from amplifying
// the rounding of the individual terms.  Sums over the tokens of
// the CTA go to shared memory (warp shuffles first); du is written as bf16.
__device__ __forceinline__ void chain_rule16(uint32_t trow, int fh, int ch, int h, int64_t tpos,
                                             bool valid, const __nv_bfloat16* urow,
                                             const BwdParams& prm, __nv_bfloat16* durow,
                                             Misc& m, int lane) {
  const float gam = prm.gamma[h];
  float du[16];
  float dgam = 0.f;
  uint4 raw[2];
  raw[0] = valid ? ldg_nc_v4(urow + 32 * fh + 16 * ch) : make_uint4(0u, 0u, 0u, 0u);
  raw[1] = valid ? ldg_nc_v4(urow + 32 * fh + 16 * ch + 8) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int gi = 0; gi < 2; ++gi) {
    const int agl = 2 * ch + gi;   // dimension group inside the half
    float dphi_ch[40];   // exactly the group's 40 columns
    tmem_ld16(trow + 40 * agl, *reinterpret_cast<float(*)[16]>(&dphi_ch[0]));
    tmem_ld16(trow + 40 * agl + 16, *reinterpret_cast<float(*)[16]>(&dphi_ch[16]));
    tmem_ld8(trow + 40 * agl + 32, *reinterpret_cast<float(*)[8]>(&dphi_ch[32]));
    tmem_ld_wait();
    const uint32_t w[4] = {raw[gi].x, raw[gi].y, raw[gi].z, raw[gi].w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int a = 32 * fh + 8 * agl + e;   // dimension
      const float u = __uint_as_float((e & 1) ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16));
      const float inv = 1.0f / (1.0f + fabsf(u));
      const float th = kPi * u * inv;
      float sx, cx;
      sincosf(th + prm.omega[h * kD + a], &sx, &cx);
      const float g = cx - sx;
      const float gp = -sx - cx;
      const float r = tanhf(gam * g);
      float sr, cr;
      sincosf(th + phase_mod_2pi(tpos, prm.phi[h * kD + a]), &sr, &cr);
      const float d1 = dphi_ch[e], d2 = dphi_ch[8 + e], d3 = dphi_ch[16 + e];
      const float d4 = dphi_ch[24 + e], d5 = dphi_ch[32 + e];
      const float dc = fmaf(r, d4, d1);
      const float ds = fmaf(r, d5, d2);
      const float dr = fmaf(sr, d5, fmaf(cr, d4, d3));
      const float dthr = fmaf(cr, ds, -sr * dc);
      const float dpre = valid ? dr * (1.0f - r * r) : 0.f;
      const float dtheta = fmaf(dpre * gam, gp, dthr);
      du[8 * gi + e] = dtheta * kPi * inv * inv;
      dgam = fmaf(dpre, g, dgam);
      float om = dpre * gam * gp;
      float ph = valid ? dthr * static_cast<float>(tpos - prm.pos_mid) : 0.f;
#pragma unroll
      for (int sh = 16; sh > 0; sh >>= 1) {
        om += __shfl_xor_sync(0xffffffffu, om, sh);
        ph += __shfl_xor_sync(0xffffffffu, ph, sh);
      }
      if (lane == 0) {
        atomicAdd(&m.red_omega[a], om);
        atomicAdd(&m.red_phi[a], ph);
      }
    }
  }
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) dgam += __shfl_xor_sync(0xffffffffu, dgam, sh);
  if (lane == 0) atomicAdd(&m.red_gamma, dgam);
  if (valid) {
    uint4 o0, o1;
    o0.x = pack_bf16x2(du[0], du[1]);   o0.y = pack_bf16x2(du[2], du[3]);
    o0.z = pack_bf16x2(du[4], du[5]);   o0.w = pack_bf16x2(du[6], du[7]);
    o1.x = pack_bf16x2(du[8], du[9]);   o1.y = pack_bf16x2(du[10], du[11]);
    o1.z = pack_bf16x2(du[12], du[13]); o1.w = pack_bf16x2(du[14], du[15]);
    uint4* dst = reinterpret_cast<uint4*>(durow + 32 * fh + 16 * ch);
    dst[0] = o0;
    dst[1] = o1;
  }
}

// Adds the CTA's shares of dgamma, domega, dphi to the outputs (after every
// epilogue thread has contributed).
__device__ __forceinline__ void flush_param_grads(const Misc& m, const BwdParams& prm, int h,
                                                  int tid) {
  if (tid < 64) {
    atomicAdd(&prm.domega[h * kD + tid], m.red_omega[tid]);
    if (prm.dphi != nullptr) atomicAdd(&prm.dphi[h * kD + tid], m.red_phi[tid]);
  }
  if (tid == 0) atomicAdd(&prm.dgamma[h], m.red_gamma);
}

// (sequence, chunk) of CTA b: groups of kSeqGroup sequences, within a group
// the heaviest chunks first (query pass: late query chunks; key pass: early
// key chunks), groups from the last sequence down.
__device__ __forceinline__ void cta_chunk(int b, int bhn, int nchunks, bool late_first, int& bh,
                                          int& chunk) {
  const int gf = min(kSeqGroup, bhn);
  const int grp = b / (gf * nchunks);
  const int gsz = min(gf, bhn - grp * gf);
  const int r = b - grp * gf * nchunks;
  chunk = late_first ? nchunks - 1 - r / gsz : r / gsz;
  bh = bhn - 1 - (grp * gf + r % gsz);
}

// Score-gradient (and weight) pairs of 32 keys: ds = (dw + dd) p x^(p-1) / 4d
// with x = (s + 64) / 4d; elements with keep(i) false get 0.  Written as bf16
// hi (truncated) + lo (rounded rest) pairs, element 2i and 2i + 1 in word i.
template <int P, typename Keep>
__device__ __forceinline__ void grads32(const float* sv, const float* dwv, const float* dd,
                                        Keep keep, uint32_t (&dhi)[16], uint32_t (&dlo)[16],
                                        uint32_t (&whi)[16], uint32_t (&wlo)[16]) {
  constexpr float kInv4d = 1.0f / (4.0f * kD);
  constexpr float kConst = 64.0f * kInv4d;
  constexpr float kScale = static_cast<float>(P) * kInv4d;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float g2[2], w2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int k = 2 * i + e;
      const float x = fmaf(sv[k], kInv4d, kConst);
      const float xp1 = pow_int<P - 1>(x);
      const bool kp = keep(k);
      g2[e] = kp ? (dwv[k] + dd[k]) * kScale * xp1 : 0.f;
      w2[e] = kp ? xp1 * x : 0.f;
    }
    const uint32_t b0 = __float_as_uint(g2[0]), b1 = __float_as_uint(g2[1]);
    dhi[i] = __byte_perm(b0, b1, 0x7632);
    dlo[i] = pack_bf16x2(g2[0] - __uint_as_float(b0 & 0xffff0000u),
                         g2[1] - __uint_as_float(b1 & 0xffff0000u));
    const uint32_t c0 = __float_as_uint(w2[0]), c1 = __float_as_uint(w2[1]);
    whi[i] = __byte_perm(c0, c1, 0x7632);
    wlo[i] = pack_bf16x2(w2[0] - __uint_as_float(c0 & 0xffff0000u),
                         w2[1] - __uint_as_float(c1 & 0xffff0000u));
  }
}

// ---------------------------------------------------------------------------
// Query pass.  Shared memory: Phi(Q_i) and dN_i resident; Phi(K) and
// [V | 1 | 0] halves streamed through two buffers.
constexpr int kQOffQ = 0;
constexpr int kQOffDN = kQOffQ + kPhiBytes;
constexpr int kQOffK = kQOffDN + kDNBytes;           // two halves
constexpr int kQOffV = kQOffK + 2 * kHalfPhi;        // two halves
constexpr int kQOffMisc = kQOffV + 2 * kHalfV;
constexpr int kQSmem = kQOffMisc + static_cast<int>(sizeof(Misc));
static_assert(kQSmem <= 232448, "query pass: shared memory exceeds 227 KB");

__device__ __forceinline__ void bulk_load_pieces(uint32_t sdst, const unsigned char* src,
                                                 uint32_t bytes, uint64_t* bar) {
  for (uint32_t off = 0; off < bytes; off += 16384)
    bulk_load_g2s(sdst + off, src + off, min(16384u, bytes - off), bar);
}

template <int P>
__global__ void __launch_bounds__(kThreads, 1) pow_bwd_q_kernel(BwdParams prm) {
  extern __shared__ __align__(1024) unsigned char smem[];
  Misc& m = *reinterpret_cast<Misc*>(smem + kQOffMisc);
  const uint32_t sQ = smem_u32(smem + kQOffQ), sDN = smem_u32(smem + kQOffDN);
  const uint32_t sK = smem_u32(smem + kQOffK), sV = smem_u32(smem + kQOffV);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bh, qi;
  cta_chunk(static_cast<int>(blockIdx.x), prm.bhn, prm.nchunks, true, bh, qi);
  const int h = bh % prm.H;
  const int ntiles = 2 * (qi + 1);   // 64-key halves of the key chunks 0..qi

  if (warp == kMmaWarp) {
    tmem_alloc(&m.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b) {
      const bool epi = b == kSFree || b == kDSReady;
      mbar_init(&m.bar[b], epi ? static_cast<uint32_t>(kEpiWarps) : 1u);
    }
    m.abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < 64) { m.red_omega[tid] = 0.f; m.red_phi[tid] = 0.f; }
  if (tid == 0) m.red_gamma = 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (warp == kLoadWarp) {
    if (lane == 0) {
      const unsigned char* cq = chunk_base(prm.ws, bh, prm.nchunks, qi);
      const unsigned char* dq = prm.dn + (static_cast<int64_t>(bh) * prm.nchunks + qi) * kDNBytes;
      mbar_arrive_expect_tx(&m.bar[kResFull], kPhiBytes + kDNBytes);
      bulk_load_pieces(sQ, cq, kPhiBytes, &m.bar[kResFull]);
      bulk_load_g2s(sDN, dq, kDNBytes, &m.bar[kResFull]);
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int b = t & 1;
        // buffer b is free once the tile that used it before has completed
        if (t >= 2 && !wait_bar(m, kTileDone0 + b, ((t - 2) >> 1) & 1)) break;
        const unsigned char* cj = chunk_base(prm.ws, bh, prm.nchunks, t >> 1);
        const uint32_t hk = static_cast<uint32_t>(t & 1);
        mbar_arrive_expect_tx(&m.bar[kStrFull0 + b], kHalfPhi + kHalfV);
        bulk_load_pieces(sK + b * kHalfPhi, cj + kPhiBytes + hk * kHalfPhi, kHalfPhi,
                         &m.bar[kStrFull0 + b]);
        bulk_load_g2s(sV + b * kHalfV, cj + 2 * kPhiBytes + hk * kHalfV, kHalfV,
                      &m.bar[kStrFull0 + b]);
        issued = t + 1;
      }
      // no copy may still be writing shared memory when the CTA exits
      mbar_wait_bounded(&m.bar[kResFull], 0, kWaitNs);
      for (int t = max(0, issued - 2); t < issued; ++t)
        mbar_wait_bounded(&m.bar[kStrFull0 + (t & 1)], (t >> 1) & 1, kWaitNs);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t idF = idesc_bf16_f32(128, 160, false, true);
      // dPhi(Q_i) += dS(t) Phi(K half of tile t): K = 64 keys, N = 2 x 160 features
      auto issue_feature_grad = [&](int t) -> bool {
        if (!wait_bar(m, kDSReady, t & 1)) return false;
        tc_fence_after();
        uint64_t dKf = smem_desc(sK + (t & 1) * kHalfPhi, kXQ, 128);   // MN-major B
        asm volatile("" : "+l"(dKf));
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          const uint32_t hi = tmem + kQTDS + 32 * (st >> 1) + 8 * (st & 1);
#pragma unroll
          for (int nh = 0; nh < 2; ++nh) {
            const uint64_t bd = dKf + 160 * nh + (2 * kXQ / 16) * st;
            mma_ts(tmem + kQTF + 160 * nh, hi, bd, idF, (t | st) != 0);
            mma_ts(tmem + kQTF + 160 * nh, hi + 16, bd, idF, true);
          }
        }
        mma_commit(&m.bar[kTileDone0 + (t & 1)]);
        return true;
      };
      bool ok = wait_bar(m, kResFull, 0);
      for (int t = 0; ok && t < ntiles; ++t) {
        const int b = t & 1;
        if (!wait_bar(m, kStrFull0 + b, (t >> 1) & 1)) break;
        // the epilogue has read the previous scores and dW from TMEM
        if (t > 0 && !wait_bar(m, kSFree, (t - 1) & 1)) break;
        tc_fence_after();
        uint64_t dQ = smem_desc(sQ, 128, kXQ);                   // Phi(Q_i), K-major A
        uint64_t dK = smem_desc(sK + b * kHalfPhi, 128, kXQ);    // Phi(K half), K-major B
        uint64_t dN = smem_desc(sDN, 128, 1024);                 // dN_i, K-major A
        uint64_t dV = smem_desc(sV + b * kHalfV, 128, kVGroup);  // V half, K-major B
        asm volatile("" : "+l"(dQ), "+l"(dK), "+l"(dN), "+l"(dV));
#pragma unroll
        for (int st = 0; st < 20; ++st)
          mma_ss(tmem + kQTS, dQ + 16 * st, dK + 16 * st, idS, st > 0);
#pragma unroll
        for (int st = 0; st < 4; ++st)
          mma_ss(tmem + kQTDW, dN + 16 * st, dV + 16 * st, idS, st > 0);
        mma_commit(&m.bar[kSDone]);
        if (t > 0 && !issue_feature_grad(t - 1)) { ok = false; break; }
        if (t == ntiles - 1) ok = issue_feature_grad(t);
      }
      // wait (bounded) for every MMA issued, also after an abandoned wait
      mma_commit(&m.bar[kDrain]);
      mbar_wait_bounded(&m.bar[kDrain], 0, kWaitNs);
    }
  } else {
    // epilogue: warp (qd, cw) owns query rows 32 qd .. + 31 and keys 32 cw .. + 31
    // of each 64-key half
    const int qd = warp & 3, cw = warp >> 2;
    const int row = 32 * qd + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
    const float ddrow = prm.dd[(static_cast<int64_t>(bh) * prm.nchunks + qi) * kC + row];
    float ddv[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) ddv[k] = ddrow;
    for (int t = 0; t < ntiles; ++t) {
      if (!wait_bar(m, kSDone, t & 1)) break;
      tc_fence_after();
      const bool diag = (t >> 1) == qi;
      const int blk = 2 * (t & 1) + cw;   // 32-key block of the chunk
      const bool none = diag && blk > qd;  // every key of the block is after every row
      float sv[32], dwv[32];
      if (!none) {
        tmem_ld16(tmem + lane_off + kQTS + 32 * cw, *reinterpret_cast<float(*)[16]>(&sv[0]));
        tmem_ld16(tmem + lane_off + kQTS + 32 * cw + 16, *reinterpret_cast<float(*)[16]>(&sv[16]));
        tmem_ld16(tmem + lane_off + kQTDW + 32 * cw, *reinterpret_cast<float(*)[16]>(&dwv[0]));
        tmem_ld16(tmem + lane_off + kQTDW + 32 * cw + 16,
                  *reinterpret_cast<float(*)[16]>(&dwv[16]));
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&m.bar[kSFree]);   // the next half's MMAs may overwrite them
      uint32_t dhi[16], dlo[16], whi[16], wlo[16];
      if (none) {
#pragma unroll
        for (int i = 0; i < 16; ++i) { dhi[i] = 0u; dlo[i] = 0u; }
      } else {
        const int lim = (diag && blk == qd) ? lane : 31;   // keys up to the row's own
        grads32<P>(sv, dwv, ddv, [lim](int k) { return k <= lim; }, dhi, dlo, whi, wlo);
      }
      // the previous half's feature-gradient MMAs have read the dS buffer
      if (t > 0 && !wait_bar(m, kTileDone0 + ((t - 1) & 1), ((t - 1) >> 1) & 1)) break;
      tc_fence_after();
      tmem_st16(tmem + lane_off + kQTDS + 32 * cw, dhi);
      tmem_st16(tmem + lane_off + kQTDS + 32 * cw + 16, dlo);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&m.bar[kDSReady]);
    }
    wait_bar(m, kTileDone0 + ((ntiles - 1) & 1), ((ntiles - 1) >> 1) & 1);
    tc_fence_after();
    const int t = qi * kC + row;
    const bool valid = t < prm.T;
    const int64_t grow = static_cast<int64_t>(bh) * prm.T + (valid ? t : 0);
#pragma unroll 1
    for (int ch = 0; ch < 2; ++ch)
      chain_rule16(tmem + lane_off + kQTF + 160 * cw, cw, ch, h, prm.pos0 + t, valid,
                   prm.u + grow * kD, prm, prm.du + grow * kD, m, lane);
    epi_sync();
    flush_param_grads(m, prm, h, tid);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Key pass.  Shared memory: Phi(K_j) and [V_j | 1 | 0] resident; Phi(Q), dN
// and dD halves streamed through two buffers.
constexpr int kKOffK = 0;
constexpr int kKOffV = kKOffK + kPhiBytes;
constexpr int kKOffQ = kKOffV + kVBytes;             // two halves
constexpr int kKOffDN = kKOffQ + 2 * kHalfPhi;       // two halves
constexpr int kKOffDD = kKOffDN + 2 * kHalfDN;       // two halves
constexpr int kKOffMisc = kKOffDD + 2 * kHalfDD;
constexpr int kKSmem = kKOffMisc + static_cast<int>(sizeof(Misc));
static_assert(kKSmem <= 232448, "key pass: shared memory exceeds 227 KB");

template <int P>
__global__ void __launch_bounds__(kThreads, 1) pow_bwd_k_kernel(BwdParams prm) {
  extern __shared__ __align__(1024) unsigned char smem[];
  Misc& m = *reinterpret_cast<Misc*>(smem + kKOffMisc);
  const float* sdd = reinterpret_cast<const float*>(smem + kKOffDD);
  const uint32_t sK = smem_u32(smem + kKOffK), sV = smem_u32(smem + kKOffV);
  const uint32_t sQ = smem_u32(smem + kKOffQ), sDN = smem_u32(smem + kKOffDN);
  const uint32_t sDD = smem_u32(smem + kKOffDD);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bh, kj;
  cta_chunk(static_cast<int>(blockIdx.x), prm.bhn, prm.nchunks, false, bh, kj);
  const int h = bh % prm.H;
  const int ntiles = 2 * (prm.nchunks - kj);   // 64-query halves of the chunks kj..

  if (warp == kMmaWarp) {
    tmem_alloc(&m.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b)
      mbar_init(&m.bar[b], b == kDSReady ? static_cast<uint32_t>(kEpiWarps) : 1u);
    m.abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < 64) { m.red_omega[tid] = 0.f; m.red_phi[tid] = 0.f; }
  if (tid == 0) m.red_gamma = 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (warp == kLoadWarp) {
    if (lane == 0) {
      const unsigned char* ck = chunk_base(prm.ws, bh, prm.nchunks, kj);
      mbar_arrive_expect_tx(&m.bar[kResFull], kPhiBytes + kVBytes);
      bulk_load_pieces(sK, ck + kPhiBytes, kPhiBytes, &m.bar[kResFull]);
      bulk_load_g2s(sV, ck + 2 * kPhiBytes, kVBytes, &m.bar[kResFull]);
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int b = t & 1;
        if (t >= 2 && !wait_bar(m, kTileDone0 + b, ((t - 2) >> 1) & 1)) break;
        const int qi = kj + (t >> 1);
        const uint32_t hq = static_cast<uint32_t>(t & 1);
        const unsigned char* cq = chunk_base(prm.ws, bh, prm.nchunks, qi);
        const int64_t sc = static_cast<int64_t>(bh) * prm.nchunks + qi;
        mbar_arrive_expect_tx(&m.bar[kStrFull0 + b], kHalfPhi + kHalfDN + kHalfDD);
        bulk_load_pieces(sQ + b * kHalfPhi, cq + hq * kHalfPhi, kHalfPhi, &m.bar[kStrFull0 + b]);
        bulk_load_g2s(sDN + b * kHalfDN, prm.dn + sc * kDNBytes + hq * kHalfDN, kHalfDN,
                      &m.bar[kStrFull0 + b]);
        bulk_load_g2s(sDD + b * kHalfDD, prm.dd + sc * kC + 64 * hq, kHalfDD,
                      &m.bar[kStrFull0 + b]);
        issued = t + 1;
      }
      mbar_wait_bounded(&m.bar[kResFull], 0, kWaitNs);
      for (int t = max(0, issued - 2); t < issued; ++t)
        mbar_wait_bounded(&m.bar[kStrFull0 + (t & 1)], (t >> 1) & 1, kWaitNs);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t idF = idesc_bf16_f32(128, 160, false, true);
      constexpr uint32_t idV = idesc_bf16_f32(128, 64, false, true);
      bool ok = wait_bar(m, kResFull, 0);
      for (int t = 0; ok && t < ntiles; ++t) {
        const int b = t & 1;
        if (!wait_bar(m, kStrFull0 + b, (t >> 1) & 1)) break;
        // the previous half's MMAs have read W^T and dS^T from the score columns
        if (t > 0 && !wait_bar(m, kTileDone0 + ((t - 1) & 1), ((t - 1) >> 1) & 1)) break;
        tc_fence_after();
        uint64_t dK = smem_desc(sK, 128, kXQ);                    // Phi(K_j), K-major A
        uint64_t dQ = smem_desc(sQ + b * kHalfPhi, 128, kXQ);     // Phi(Q half), K-major B
        uint64_t dV = smem_desc(sV, 128, kVGroup);                // V_j, K-major A
        uint64_t dN = smem_desc(sDN + b * kHalfDN, 128, 1024);    // dN half, K-major B
        asm volatile("" : "+l"(dK), "+l"(dQ), "+l"(dV), "+l"(dN));
#pragma unroll
        for (int st = 0; st < 20; ++st)
          mma_ss(tmem + kKTS, dK + 16 * st, dQ + 16 * st, idS, st > 0);
#pragma unroll
        for (int st = 0; st < 4; ++st)
          mma_ss(tmem + kKTDW, dV + 16 * st, dN + 16 * st, idS, st > 0);
        mma_commit(&m.bar[kSDone]);
        if (!wait_bar(m, kDSReady, t & 1)) break;
        tc_fence_after();
        uint64_t dQf = smem_desc(sQ + b * kHalfPhi, kXQ, 128);    // Phi(Q half), MN-major B
        uint64_t dNv = smem_desc(sDN + b * kHalfDN, 1024, 128);   // dN half, MN-major B
        asm volatile("" : "+l"(dQf), "+l"(dNv));
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          const uint32_t hs = tmem + kKTDW + 32 * (st >> 1) + 8 * (st & 1);   // dS^T
          const uint32_t hw = tmem + kKTS + 32 * (st >> 1) + 8 * (st & 1);    // W^T
#pragma unroll
          for (int nh = 0; nh < 2; ++nh) {
            const uint64_t bd = dQf + 160 * nh + (2 * kXQ / 16) * st;
            mma_ts(tmem + kKTF + 160 * nh, hs, bd, idF, (t | st) != 0);
            mma_ts(tmem + kKTF + 160 * nh, hs + 16, bd, idF, true);
          }
          const uint64_t vd = dNv + (2 * 1024 / 16) * st;
          mma_ts(tmem + kKTV, hw, vd, idV, (t | st) != 0);
          mma_ts(tmem + kKTV, hw + 16, vd, idV, true);
        }
        mma_commit(&m.bar[kTileDone0 + b]);
      }
      mma_commit(&m.bar[kDrain]);
      mbar_wait_bounded(&m.bar[kDrain], 0, kWaitNs);
    }
  } else {
    // epilogue: warp (qd, cw) owns key rows 32 qd .. + 31 and queries 32 cw .. + 31
    // of each 64-query half
    const int qd = warp & 3, cw = warp >> 2;
    const int row = 32 * qd + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
    for (int t = 0; t < ntiles; ++t) {
      const int b = t & 1;
      if (!wait_bar(m, kStrFull0 + b, (t >> 1) & 1)) break;   // dD of the half in shared memory
      if (!wait_bar(m, kSDone, t & 1)) break;
      tc_fence_after();
      const bool diag = (t >> 1) == 0;    // query chunk == key chunk
      const int qblk = 2 * (t & 1) + cw;  // 32-query block of the chunk
      uint32_t dhi[16], dlo[16], whi[16], wlo[16];
      if (diag && qblk < qd) {   // every query of the block is before every key of the warp
#pragma unroll
        for (int i = 0; i < 16; ++i) { dhi[i] = 0u; dlo[i] = 0u; whi[i] = 0u; wlo[i] = 0u; }
      } else {
        float sv[32], dwv[32];
        tmem_ld16(tmem + lane_off + kKTS + 32 * cw, *reinterpret_cast<float(*)[16]>(&sv[0]));
        tmem_ld16(tmem + lane_off + kKTS + 32 * cw + 16, *reinterpret_cast<float(*)[16]>(&sv[16]));
        tmem_ld16(tmem + lane_off + kKTDW + 32 * cw, *reinterpret_cast<float(*)[16]>(&dwv[0]));
        tmem_ld16(tmem + lane_off + kKTDW + 32 * cw + 16,
                  *reinterpret_cast<float(*)[16]>(&dwv[16]));
        tmem_ld_wait();
        const int first = (diag && qblk == qd) ? lane : 0;   // queries from the key's own
        grads32<P>(sv, dwv, sdd + b * 64 + 32 * cw, [first](int k) { return k >= first; }, dhi,
                   dlo, whi, wlo);
      }
      tmem_st16(tmem + lane_off + kKTS + 32 * cw, whi);
      tmem_st16(tmem + lane_off + kKTS + 32 * cw + 16, wlo);
      tmem_st16(tmem + lane_off + kKTDW + 32 * cw, dhi);
      tmem_st16(tmem + lane_off + kKTDW + 32 * cw + 16, dlo);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&m.bar[kDSReady]);
    }
    wait_bar(m, kTileDone0 + ((ntiles - 1) & 1), ((ntiles - 1) >> 1) & 1);
    tc_fence_after();
    const int t = kj * kC + row;
    const bool valid = t < prm.T;
    const int64_t grow = static_cast<int64_t>(bh) * prm.T + (valid ? t : 0);
    {
      float dvv[32];
      tmem_ld16(tmem + lane_off + kKTV + 32 * cw, *reinterpret_cast<float(*)[16]>(&dvv[0]));
      tmem_ld16(tmem + lane_off + kKTV + 32 * cw + 16, *reinterpret_cast<float(*)[16]>(&dvv[16]));
      tmem_ld_wait();
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(prm.dv + grow * kD + 32 * cw);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          dst[q4] = make_uint4(pack_bf16x2(dvv[8 * q4], dvv[8 * q4 + 1]),
                               pack_bf16x2(dvv[8 * q4 + 2], dvv[8 * q4 + 3]),
                               pack_bf16x2(dvv[8 * q4 + 4], dvv[8 * q4 + 5]),
                               pack_bf16x2(dvv[8 * q4 + 6], dvv[8 * q4 + 7]));
      }
    }
#pragma unroll 1
    for (int ch = 0; ch < 2; ++ch)
      chain_rule16(tmem + lane_off + kKTF + 160 * cw, cw, ch, h, prm.pos0 + t, valid,
                   prm.u + grow * kD, prm, prm.du + grow * kD, m, lane);
    epi_sync();
    flush_param_grads(m, prm, h, tid);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t pow_bwd_tc_workspace_bytes(int B, int H, int T) {
  const int64_t nchunks = (static_cast<int64_t>(T) + kC - 1) / kC;
  return static_cast<size_t>(B) * H * nchunks * (kChunkBytes + kDNBytes + kDDBytes);
}

namespace {
constexpr int kMaxP = 8;
using BwdKernel = void (*)(BwdParams);

BwdKernel q_kernel_for(int p) {
  switch (p) {
    case 1: return pow_bwd_q_kernel<1>;
    case 2: return pow_bwd_q_kernel<2>;
    case 3: return pow_bwd_q_kernel<3>;
    case 4: return pow_bwd_q_kernel<4>;
    case 5: return pow_bwd_q_kernel<5>;
    case 6: return pow_bwd_q_kernel<6>;
    case 7: return pow_bwd_q_kernel<7>;
    default: return pow_bwd_q_kernel<8>;
  }
}

BwdKernel k_kernel_for(int p) {
  switch (p) {
    case 1: return pow_bwd_k_kernel<1>;
    case 2: return pow_bwd_k_kernel<2>;
    case 3: return pow_bwd_k_kernel<3>;
    case 4: return pow_bwd_k_kernel<4>;
    case 5: return pow_bwd_k_kernel<5>;
    case 6: return pow_bwd_k_kernel<6>;
    case 7: return pow_bwd_k_kernel<7>;
    default: return pow_bwd_k_kernel<8>;
  }
}

cudaError_t bwd_set_smem() {
  static bool done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  for (int p = 1; p <= kMaxP && e == cudaSuccess; ++p) {
    e = cudaFuncSetAttribute(q_kernel_for(p), cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_kernel_for(p), cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kKSmem);
  }
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}
}  // namespace

cudaError_t pow_bwd_tc_launch(const PowBwdArgs& a, cudaStream_t st) {
  const PowFwdArgs& f = a.f;
  const int bhn = f.B * f.H;
  const int nchunks = (f.T + kC - 1) / kC;
  cudaError_t e;
  // the parameter gradients are sums: start from zero
  if (f.H > 0) {
    if ((e = cudaMemsetAsync(a.dgamma, 0, sizeof(float) * f.H, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.domega, 0, sizeof(float) * f.H * kD, st)) != cudaSuccess) return e;
    if (a.dphi != nullptr &&
        (e = cudaMemsetAsync(a.dphi, 0, sizeof(float) * f.H * kD, st)) != cudaSuccess)
      return e;
  }
  if (bhn == 0 || nchunks == 0) return cudaSuccess;
  if (f.p < 1 || f.p > kMaxP) return cudaErrorInvalidValue;
  if ((e = bwd_set_smem()) != cudaSuccess) return e;
  unsigned char* ws = static_cast<unsigned char*>(f.workspace);
  const int64_t nsc = static_cast<int64_t>(bhn) * nchunks;
  unsigned char* dn = ws + nsc * kChunkBytes;
  float* dd = reinterpret_cast<float*>(dn + nsc * kDNBytes);
  if ((e = pow_prep_launch(f, st)) != cudaSuccess) return e;
  DPrepParams dp{};
  dp.dO = a.dO;
  dp.grad_bf16 = a.grad_dtype == SANATAN_BF16;
  dp.o = a.o;
  dp.D = a.D;
  dp.eps = f.eps;
  dp.T = f.T;
  dp.nchunks = nchunks;
  dp.ntok = nsc * kC;
  dp.dn = dn;
  dp.dd = dd;
  const int64_t threads = dp.ntok * 8;
  pow_dprep_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(dp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  BwdParams bp{};
  bp.ws = ws;
  bp.dn = dn;
  bp.dd = dd;
  bp.gamma = f.gamma;
  bp.omega = f.omega;
  bp.phi = f.phi;
  bp.H = f.H;
  bp.T = f.T;
  bp.nchunks = nchunks;
  bp.bhn = bhn;
  bp.pos0 = f.pos0;
  bp.pos_mid = f.pos0 + (f.T - 1) / 2;
  bp.dgamma = a.dgamma;
  bp.domega = a.domega;
  bp.dphi = a.dphi;
  const unsigned grid = static_cast<unsigned>(nsc);
  bp.u = static_cast<const __nv_bfloat16*>(f.q);
  bp.du = static_cast<__nv_bfloat16*>(a.dq);
  bp.dv = nullptr;
  q_kernel_for(f.p)<<<grid, kThreads, kQSmem, st>>>(bp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bp.u = static_cast<const __nv_bfloat16*>(f.k);
  bp.du = static_cast<__nv_bfloat16*>(a.dk);
  bp.dv = static_cast<__nv_bfloat16*>(a.dv);
  const ProfileEvents& pe = profile_events();
  const bool rec = pe.start != nullptr;
  if (rec) cudaEventRecord(pe.start, st);
  k_kernel_for(f.p)<<<grid, kThreads, kKSmem, st>>>(bp);
  e = cudaGetLastError();
  if (rec) cudaEventRecord(pe.stop, st);
  return e;
}

int pow_bwd_tc_read_and_clear_error(cudaStream_t st) {
  int h = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_pow_bwd_error, sizeof(int), 0, cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return -1;
  if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_pow_bwd_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                st) != cudaSuccess)
      return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  }
  return h;
}

}  // namespace sanatan
