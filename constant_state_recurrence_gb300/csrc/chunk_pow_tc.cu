// Power-sharpened causal attention on the tensor cores (bf16 operands, f32
// accumulation): eq. (8) of "SANATAN: Root-Parity Gated Angular Attention with
// an Exact Constant-State Recurrent Form" (reading notes §2.6) at a positive
// integer power p,
//   a_tj = (s_tj / 4d)^p / (sum_{l<=t} (s_tl / 4d)^p + eps),  o_t = sum_{j<=t} a_tj v_j,
// with s_tj = Phi(q_t).Phi(k_j).  For p > 1 there is no small state (the
// notes: the tensor-power features grow as (6d)^p), so this is the parallel
// quadratic form the paper trains with.
//
// Two kernels.  The preparation kernel featurises q and k once (the bf16
// feature map of the recurrent path) and writes Phi(Q), Phi(K) and [V | 1 | 0]
// chunk by chunk in the operand layouts, so the attention kernel fetches each
// 128-token chunk with plain bulk copies.  The attention kernel runs one CTA
// per (sequence, query chunk): Phi(Q) is copied once into TMEM and is the A
// operand of every score product; for every key chunk j up to the diagonal,
// P = Phi(Q) Phi(K_j)^T (M = N = 128, K = 320) lands in one of two TMEM
// buffers, the epilogue raises (P + 64) / 4d to the power p (64 is the
// constant channel's exact contribution), masks the diagonal chunk and
// splits the weights into bf16 hi + lo halves in place, and
// O += P~ [V_j | 1 | 0] (`.ts`, N = 80) accumulates the outputs and, in the
// ones column, the denominator.  Heavy (late) query chunks are scheduled
// first.
#include "sanatan_internal.h"
#include "sanatan_math.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"
#include "pow_common.cuh"

namespace sanatan {

__device__ int g_pow_tc_error;  // set when a bounded wait gives up

namespace {

using namespace tc;
using namespace tcc;
using namespace powc;

// Shared memory: two Phi(K) and two V buffers (chunk j uses buffer j & 1).
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + 2 * kPhiBytes;
constexpr int kOffMisc = kOffV + 2 * kVBytes;

// TMEM columns: two score buffers, the output accumulator, and Phi(Q) as the
// A operand of the score products (320 bf16 features = 160 columns; column
// 4 fg + p holds dimensions 2p, 2p + 1 of feature group fg).
constexpr uint32_t kTP0 = 0;      // score buffers at 0 and 128
constexpr uint32_t kTO = 256;     // output accumulator [O | denominator | 0] (80 columns)
constexpr uint32_t kTQ = 352;     // Phi(Q)
constexpr uint32_t kTmemCols = 512;

enum Bar {
  kQReady = 0, kKFull0, kKFull1, kKFree0, kKFree1, kVFull0, kVFull1, kPFull0, kPFull1,
  kPTilde0, kPTilde1, kPVDone0, kPVDone1, kODone, kNumBars
};

struct Misc {
  uint64_t bar[kNumBars];
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int kSmemBytes = kOffMisc + static_cast<int>(sizeof(Misc));
static_assert(kSmemBytes <= 232448, "shared memory layout exceeds 227 KB");

// warps 0-7 epilogue (warp w: TMEM lanes 32 (w % 4) .. +31, key columns
// 64 (w / 4) .. +63), warp 8 MMA issue, warp 9 Phi(K) loads, warp 10 V loads
constexpr int kEpiWarps = 8;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kVLoadWarp = 10;
constexpr int kThreads = 32 * (kVLoadWarp + 1);
constexpr uint64_t kWaitNs = 2000000000ull;

struct PowParams {
  const unsigned char* ws;   // per (sequence, chunk): Phi(Q) | Phi(K) | V
  int H, T, nchunks, bhn;
  float eps;
  float inv_c;               // ablation maps: 1 / (score scale)
  float cst;                 // ablation maps: (d + shift) / scale, the constant channel and shift
  float* o;                  // [B, H, T, 64] f32
  float* Dn;                 // [B, H, T] f32 or null
};

struct PrepParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* gamma;
  const float* omega;
  const float* phi;
  int H, T, nchunks;
  int64_t pos0;
  unsigned char* ws;
};

// ---------------------------------------------------------------------------
// Preparation: one CTA of 256 threads per half chunk (64 tokens).  Lane
// (r, dimension group ag) of warp w owns the chunk's tokens tq + 8 i (i < 2),
// tq = 64 half + 16 (w / 2) + r.
// CH = 6: the six-channel map; CH = 4 / 3: the ablation maps, whose CH - 1
// non-constant channels fill feature groups (CH - 1) ag + c - 1 of the same
// chunk layout (the rest of a chunk's feature groups is not read).
constexpr int kPrepTok = 2;
template <int CH>
__global__ void __launch_bounds__(256) pow_prep_kernel(PrepParams prm) {
  __shared__ float4 dimc[64];
  const int half = blockIdx.x & 1;
  const int bh = (blockIdx.x >> 1) / prm.nchunks;
  const int chunk = (blockIdx.x >> 1) % prm.nchunks;
  const int h = bh % prm.H;
  const int tid = threadIdx.x;
  if (tid < kD) {
    const float g = prm.gamma[h] * 1.41421356237309515f;
    float sw, cw;
    sincosf(prm.omega[h * kD + tid] + 0.785398163397448310f, &sw, &cw);
    float s8, c8;
    sincosf(phase_mod_2pi(8, prm.phi[h * kD + tid]), &s8, &c8);
    dimc[tid] = make_float4(g * cw, g * sw, c8, s8);
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  const int r = lane & 7;
  const int ag = (lane >> 3) + 4 * (warp & 1);
  const int tq = 64 * half + 16 * (warp >> 1) + r;
  const int tok0 = chunk * kC;
  const int64_t seq_row0 = static_cast<int64_t>(bh) * prm.T;
  unsigned char* base = prm.ws + (static_cast<int64_t>(bh) * prm.nchunks + chunk) * kChunkBytes;
  // every load of the thread first (q, k, v of its tokens), then the math
  uint4 raw[3][kPrepTok];
#pragma unroll
  for (int w = 0; w < 3; ++w) {
    const __nv_bfloat16* src = w == 0 ? prm.q : (w == 1 ? prm.k : prm.v);
#pragma unroll
    for (int i = 0; i < kPrepTok; ++i) {
      const int t = tq + 8 * i;
      raw[w][i] = (tok0 + t < prm.T) ? ldg_nc_v4(src + (seq_row0 + tok0 + t) * kD + 8 * ag)
                                     : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // V: 8 columns (group ag) of each of the thread's tokens (zero past the end)
  unsigned char* vdst = base + 2 * kPhiBytes;
#pragma unroll
  for (int i = 0; i < kPrepTok; ++i) {
    const int t = tq + 8 * i;
    unsigned char* vrow = vdst + (t >> 3) * kVGroup + (t & 7) * 16;
    *reinterpret_cast<uint4*>(vrow + ag * 128) = raw[2][i];
    if (ag == 0) {  // the ones column (bf16 1.0) and its zero padding
      *reinterpret_cast<uint4*>(vrow + 8 * 128) = make_uint4(0x3F80u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(vrow + 9 * 128) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  const float4* dc = &dimc[8 * ag];
  float cb0[8], sb0[8];
  {
    const int64_t tabs = prm.pos0 + tok0 + tq;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      __sincosf(phase_mod_2pi(tabs, prm.phi[h * kD + 8 * ag + j]), &sb0[j], &cb0[j]);
  }
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    unsigned char* dst = base + which * kPhiBytes;
    float cb[8], sb[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) { cb[j] = cb0[j]; sb[j] = sb0[j]; }
#pragma unroll
    for (int i = 0; i < kPrepTok; ++i) {
      const int t = tq + 8 * i;
      const bool valid = tok0 + t < prm.T;
      if constexpr (CH == 6) {
        uint32_t f[5][4];
        if (valid) {
          features8(raw[which][i], dc, cb, sb, f);
        } else {
#pragma unroll
          for (int c = 0; c < 5; ++c)
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) f[c][pp] = 0u;
        }
#pragma unroll
        for (int c = 0; c < 5; ++c)
          *reinterpret_cast<uint4*>(dst + phi_offset(t, feat_group(ag, c + 1))) =
              make_uint4(f[c][0], f[c][1], f[c][2], f[c][3]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 kc = dc[j];
          const float nc = fmaf(cb[j], kc.z, -sb[j] * kc.w);
          sb[j] = fmaf(sb[j], kc.z, cb[j] * kc.w);
          cb[j] = nc;
        }
      } else {
        uint32_t f[CH - 1][4];
        features8_map<CH>(raw[which][i], dc, cb, sb, f);  // raw is zero past the end
#pragma unroll
        for (int c = 0; c < CH - 1; ++c)
          *reinterpret_cast<uint4*>(dst + phi_offset(t, (CH - 1) * ag + c)) =
              valid ? make_uint4(f[c][0], f[c][1], f[c][2], f[c][3]) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
}

__device__ __forceinline__ bool wait_bar(Misc& m, int b, uint32_t parity) {
  if (*reinterpret_cast<volatile int*>(&m.abort_flag)) return false;
  if (mbar_wait_bounded(&m.bar[b], parity, kWaitNs)) return true;
  m.abort_flag = 1;
  atomicOr(&g_pow_tc_error, 1);
  return false;
}

// The weights ((s / 4d)^p) of 32 keys of one row from their scores,
// split into bf16 pairs hi (the truncated value) + lo (the rounded rest), keys
// 2i and 2i + 1 in word i.  MASK: keys after `lim` get weight 0.
// Packed f32x2 arithmetic (two float32 lanes in one 64-bit register; each
// lane rounds as the scalar instruction does).
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
template <int P>
__device__ __forceinline__ uint64_t pow_int2(uint64_t x) {
  if constexpr (P <= 1) {
    return x;
  } else {
    const uint64_t h = pow_int2<P / 2>(x);
    const uint64_t h2 = fmul2(h, h);
    return (P & 1) ? fmul2(h2, x) : h2;
  }
}

// The weights ((s / 4d)^p) of 32 keys of one row from their scores, split
// into bf16 pairs hi (the truncated value) + lo (the rounded rest), keys 2i and
// 2i + 1 in word i.  MASK: keys after `lim` get weight 0.  Two keys per
// packed instruction.
template <int P, bool MASK>
__device__ __forceinline__ void weights32(const float* pv, int lim, uint32_t (&hi)[16],
                                          uint32_t (&lo)[16]) {
  constexpr float kInv4d = 1.0f / (4.0f * kD);
  constexpr float kConst = 64.0f * kInv4d;   // the constant channel's share of s / 4d
  const uint64_t scale = pk2(kInv4d, kInv4d), shift = pk2(kConst, kConst);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float x0, x1;
    upk2(pow_int2<P>(ffma2(pk2(pv[2 * i], pv[2 * i + 1]), scale, shift)), x0, x1);
    if (MASK) {
      if (2 * i > lim) x0 = 0.f;
      if (2 * i + 1 > lim) x1 = 0.f;
    }
    const uint32_t b0 = __float_as_uint(x0), b1 = __float_as_uint(x1);
    hi[i] = __byte_perm(b0, b1, 0x7632);
    float r0, r1;
    upk2(fsub2(pk2(x0, x1), pk2(__uint_as_float(b0 & 0xffff0000u),
                                __uint_as_float(b1 & 0xffff0000u))), r0, r1);
    lo[i] = pack_bf16x2(r0, r1);
  }
}

// The same for an ablation map: x = max(s + d + shift, 0) / c, with s the
// non-constant part of the score (the clip matters for the four-channel map,
// whose scores can be negative).
template <int P, bool MASK>
__device__ __forceinline__ void weights32_map(const float* pv, int lim, float inv_c, float cst,
                                              uint32_t (&hi)[16], uint32_t (&lo)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float x0 = pow_int<P>(fmaxf(fmaf(pv[2 * i], inv_c, cst), 0.0f));
    float x1 = pow_int<P>(fmaxf(fmaf(pv[2 * i + 1], inv_c, cst), 0.0f));
    if (MASK) {
      if (2 * i > lim) x0 = 0.f;
      if (2 * i + 1 > lim) x1 = 0.f;
    }
    const uint32_t b0 = __float_as_uint(x0), b1 = __float_as_uint(x1);
    hi[i] = __byte_perm(b0, b1, 0x7632);
    lo[i] = pack_bf16x2(x0 - __uint_as_float(b0 & 0xffff0000u),
                        x1 - __uint_as_float(b1 & 0xffff0000u));
  }
}

template <int P, int CH, bool MASK>
__device__ __forceinline__ void weights_for(const float* pv, int lim, const PowParams& prm,
                                            uint32_t (&hi)[16], uint32_t (&lo)[16]) {
  if constexpr (CH == 6)
    weights32<P, MASK>(pv, lim, hi, lo);
  else
    weights32_map<P, MASK>(pv, lim, prm.inv_c, prm.cst, hi, lo);
}

// ---------------------------------------------------------------------------
// CH: channels per dimension of the feature map (6; 4 and 3 for the ablation
// maps, whose 8 (CH - 1) feature groups shorten the score products).
constexpr int kSeqGroup = 8;

template <int P, int CH>
__global__ void __launch_bounds__(kThreads, 1) pow_attn_kernel(PowParams prm) {
  constexpr int kNFG = 8 * (CH - 1);   // non-constant feature groups
  constexpr int kKSteps = kNFG / 2;    // K = 16 per score MMA
  extern __shared__ __align__(1024) unsigned char smem[];
  Misc& m = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const uint32_t sK = smem_u32(smem + kOffK);
  const uint32_t sV = smem_u32(smem + kOffV);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // Query chunk qi of sequence bh.  CTAs run in groups of kSeqGroup
  // sequences, within a group the late (heavier) query chunks first, so that
  // the CTAs resident at a time read the key chunks of a few sequences, which
  // stay in L2 between their readers; groups from the last sequence down (the
  // preparation kernel wrote the last ones most recently).
  const int b = static_cast<int>(blockIdx.x);
  const int gsz_full = min(kSeqGroup, prm.bhn);
  const int grp = b / (gsz_full * prm.nchunks);
  const int gsz = min(gsz_full, prm.bhn - grp * gsz_full);
  const int r = b - grp * gsz_full * prm.nchunks;
  const int qi = prm.nchunks - 1 - r / gsz;
  const int bh = prm.bhn - 1 - (grp * gsz_full + r % gsz);
  const int nk = qi + 1;

  if (warp == kMmaWarp) {
    tmem_alloc(&m.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b) {
      const bool epi = b == kQReady || b == kPTilde0 || b == kPTilde1;
      mbar_init(&m.bar[b], epi ? static_cast<uint32_t>(kEpiWarps) : 1u);
    }
    m.abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (warp == kLoadWarp) {
    // ------------------------------------------------- Phi(K) loads
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < nk; ++j) {
        const unsigned char* cj = chunk_base(prm.ws, bh, prm.nchunks, j);
        const int b = j & 1;
        // chunk j + 2 into L2 ahead of its shared-memory load
        if (j + 2 < nk) {
          const unsigned char* cn = chunk_base(prm.ws, bh, prm.nchunks, j + 2);
          prefetch_l2_bulk(cn + kPhiBytes, kPhiBytes + kVBytes);
        }
        // Phi(K_j) into buffer b once the scores of chunk j - 2 have read it;
        // after an abandoned wait nothing more is issued
        if (j >= 2 && !wait_bar(m, b ? kKFree1 : kKFree0, ((j >> 1) - 1) & 1)) break;
        mbar_arrive_expect_tx(&m.bar[b ? kKFull1 : kKFull0], kPhiBytes);
        for (uint32_t off = 0; off < kPhiBytes; off += 16384)
          bulk_load_g2s(sK + b * kPhiBytes + off, cj + kPhiBytes + off, 16384,
                        &m.bar[b ? kKFull1 : kKFull0]);
        issued = j + 1;
      }
      // No copy may still be writing shared memory when the CTA exits, even
      // after an abandoned wait: wait (bounded) for the last issued phases.
      for (int j = (issued >= 2 ? issued - 2 : 0); j < issued; ++j)
        mbar_wait_bounded(&m.bar[(j & 1) ? kKFull1 : kKFull0], (j >> 1) & 1, kWaitNs);
    }
  } else if (warp == kVLoadWarp) {
    // ------------------------------------------------- V loads
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < nk; ++j) {
        const unsigned char* cj = chunk_base(prm.ws, bh, prm.nchunks, j);
        const int b = j & 1;
        // V_j into buffer b once P~ V of chunk j - 2 is done
        if (j >= 2 && !wait_bar(m, b ? kPVDone1 : kPVDone0, ((j >> 1) - 1) & 1)) break;
        mbar_arrive_expect_tx(&m.bar[b ? kVFull1 : kVFull0], kVBytes);
        bulk_load_g2s(sV + b * kVBytes, cj + 2 * kPhiBytes, kVBytes, &m.bar[b ? kVFull1 : kVFull0]);
        issued = j + 1;
      }
      for (int j = (issued >= 2 ? issued - 2 : 0); j < issued; ++j)
        mbar_wait_bounded(&m.bar[(j & 1) ? kVFull1 : kVFull0], (j >> 1) & 1, kWaitNs);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idQK = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idPV = idesc_bf16_f32(128, kNV, false, true);
      // After an abandoned wait no further MMA is issued (the drain below
      // still waits for the ones already issued).
      bool live = wait_bar(m, kQReady, 0);
      auto issue_qk = [&](int j) {
        const int b = j & 1;
        // score buffer b is free once P~ V of chunk j - 2 is done
        if (j >= 2 && !wait_bar(m, b ? kPVDone1 : kPVDone0, ((j >> 1) - 1) & 1)) return false;
        uint64_t dk = smem_desc(sK + b * kPhiBytes, 128, kXQ);  // Phi(K_j), K-major B
        asm volatile("" : "+l"(dk));
        if (!wait_bar(m, b ? kKFull1 : kKFull0, (j >> 1) & 1)) return false;
        tc_fence_after();
#pragma unroll
        for (int st = 0; st < kKSteps; ++st)
          mma_ts(tmem + kTP0 + 128 * b, tmem + kTQ + 8 * st, dk + 16 * st, idQK, st > 0);
        mma_commit(&m.bar[b ? kKFree1 : kKFree0]);
        mma_commit(&m.bar[b ? kPFull1 : kPFull0]);
        return true;
      };
      live = live && issue_qk(0);
      for (int j = 0; j < nk && live; ++j) {
        if (j + 1 < nk && !issue_qk(j + 1)) break;
        const int b = j & 1;
        if (!wait_bar(m, b ? kPTilde1 : kPTilde0, (j >> 1) & 1)) break;
        if (!wait_bar(m, b ? kVFull1 : kVFull0, (j >> 1) & 1)) break;
        tc_fence_after();
        uint64_t dv = smem_desc(sV + b * kVBytes, kVGroup, 128);  // [V_j | 1 | 0], MN-major B
        asm volatile("" : "+l"(dv));
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          const uint32_t hi = tmem + kTP0 + 128 * b + 32 * (st >> 1) + 8 * (st & 1);
          mma_ts(tmem + kTO, hi, dv + (2 * kVGroup / 16) * st, idPV, (j | st) != 0);
          mma_ts(tmem + kTO, hi + 16, dv + (2 * kVGroup / 16) * st, idPV, true);
        }
        mma_commit(&m.bar[b ? kPVDone1 : kPVDone0]);
      }
      mma_commit(&m.bar[kODone]);
      // nothing may be in flight when TMEM is released
      mbar_wait_bounded(&m.bar[kODone], 0, kWaitNs);
    }
  } else {
    // ------------------------------------------------- epilogue (warps 0-7)
    const int qd = warp & 3;
    const int ch = warp >> 2;
    const int row = 32 * qd + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
    {
      // Phi(Q) of this row, feature groups 20 ch .. 20 ch + 19, into TMEM
      constexpr int kHalf = kNFG / 2;   // feature groups per half
      const unsigned char* src =
          chunk_base(prm.ws, bh, prm.nchunks, qi) + phi_offset(row, kHalf * ch);
      uint4 w[kHalf];
#pragma unroll
      for (int g = 0; g < kHalf; ++g) w[g] = ldg_nc_v4(src + g * 128);
#pragma unroll
      for (int s4 = 0; s4 < kHalf / 4; ++s4) {
        uint32_t r[16];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          r[4 * g] = w[4 * s4 + g].x;
          r[4 * g + 1] = w[4 * s4 + g].y;
          r[4 * g + 2] = w[4 * s4 + g].z;
          r[4 * g + 3] = w[4 * s4 + g].w;
        }
        tmem_st16(tmem + lane_off + kTQ + 4 * kHalf * ch + 16 * s4, r);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&m.bar[kQReady]);
    }
    for (int j = 0; j < nk; ++j) {
      const int b = j & 1;
      if (!wait_bar(m, b ? kPFull1 : kPFull0, (j >> 1) & 1)) break;
      tc_fence_after();
      const bool diag = (j == qi);
      const uint32_t col0 = tmem + lane_off + kTP0 + 128 * b + 64 * ch;
      float pv[64];
      if (!(diag && 2 * ch > qd)) {
        tmem_ld16(col0, *reinterpret_cast<float(*)[16]>(&pv[0]));
        tmem_ld16(col0 + 16, *reinterpret_cast<float(*)[16]>(&pv[16]));
        tmem_ld16(col0 + 32, *reinterpret_cast<float(*)[16]>(&pv[32]));
        tmem_ld16(col0 + 48, *reinterpret_cast<float(*)[16]>(&pv[48]));
        tmem_ld_wait();
      }
#pragma unroll
      for (int bi = 0; bi < 2; ++bi) {
        const int blk = 2 * ch + bi;
        uint32_t hi[16], lo[16];
        if (!diag) {
          weights_for<P, CH, false>(pv + 32 * bi, 31, prm, hi, lo);
        } else if (blk == qd) {  // keys up to the row's own
          weights_for<P, CH, true>(pv + 32 * bi, lane, prm, hi, lo);
        } else if (blk < qd) {
          weights_for<P, CH, false>(pv + 32 * bi, 31, prm, hi, lo);
        } else {  // every key of this block is after every row of this warp
#pragma unroll
          for (int i = 0; i < 16; ++i) { hi[i] = 0u; lo[i] = 0u; }
        }
        // in place: hi over keys 32 blk .. +15 of the block's own columns, lo after it
        tmem_st16(col0 + 32 * bi, hi);
        tmem_st16(col0 + 32 * bi + 16, lo);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&m.bar[b ? kPTilde1 : kPTilde0]);
    }
    wait_bar(m, kODone, 0);
    tc_fence_after();
    float ov[32], dn[16];
    tmem_ld16(tmem + lane_off + kTO + 32 * ch, *reinterpret_cast<float(*)[16]>(&ov[0]));
    tmem_ld16(tmem + lane_off + kTO + 32 * ch + 16, *reinterpret_cast<float(*)[16]>(&ov[16]));
    tmem_ld16(tmem + lane_off + kTO + 64, dn);   // the denominator column
    tmem_ld_wait();
    const float den = dn[0];
    const int t = qi * kC + row;
    if (t < prm.T) {
      const int64_t grow = static_cast<int64_t>(bh) * prm.T + t;
      const float inv = 1.0f / (den + prm.eps);
      float4* dst = reinterpret_cast<float4*>(prm.o + grow * kD + 32 * ch);
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4)
        dst[e4] = make_float4(ov[4 * e4] * inv, ov[4 * e4 + 1] * inv, ov[4 * e4 + 2] * inv,
                              ov[4 * e4 + 3] * inv);
      if (prm.Dn != nullptr && ch == 0) prm.Dn[grow] = den;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t pow_fwd_tc_workspace_bytes(int B, int H, int T) {
  const int64_t nchunks = (static_cast<int64_t>(T) + kC - 1) / kC;
  return static_cast<size_t>(B) * H * nchunks * kChunkBytes;
}

namespace {
constexpr int kMaxP = 8;
using AttnKernel = void (*)(PowParams);
AttnKernel attn_kernel_for(int p) {
  switch (p) {
    case 1: return pow_attn_kernel<1, 6>;
    case 2: return pow_attn_kernel<2, 6>;
    case 3: return pow_attn_kernel<3, 6>;
    case 4: return pow_attn_kernel<4, 6>;
    case 5: return pow_attn_kernel<5, 6>;
    case 6: return pow_attn_kernel<6, 6>;
    case 7: return pow_attn_kernel<7, 6>;
    default: return pow_attn_kernel<8, 6>;
  }
}

// Ablation maps: p in {1, 2, 4} (nullptr otherwise).
AttnKernel ablation_kernel_for(int p, int channels) {
  if (channels == 4) {
    if (p == 1) return pow_attn_kernel<1, 4>;
    if (p == 2) return pow_attn_kernel<2, 4>;
    if (p == 4) return pow_attn_kernel<4, 4>;
  } else if (channels == 3) {
    if (p == 1) return pow_attn_kernel<1, 3>;
    if (p == 2) return pow_attn_kernel<2, 3>;
    if (p == 4) return pow_attn_kernel<4, 3>;
  }
  return nullptr;
}

cudaError_t pow_set_smem() {
  static bool done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  for (int p = 1; p <= kMaxP && e == cudaSuccess; ++p)
    e = cudaFuncSetAttribute(attn_kernel_for(p), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
  for (int ch = 3; ch <= 4 && e == cudaSuccess; ++ch)
    for (int p = 1; p <= 4 && e == cudaSuccess; ++p)
      if (AttnKernel kf = ablation_kernel_for(p, ch))
        e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}
}  // namespace

cudaError_t pow_prep_launch(const PowFwdArgs& a, cudaStream_t st) {
  const int bhn = a.B * a.H;
  const int nchunks = (a.T + kC - 1) / kC;
  if (bhn == 0 || nchunks == 0) return cudaSuccess;
  PrepParams pp{};
  pp.q = static_cast<const __nv_bfloat16*>(a.q);
  pp.k = static_cast<const __nv_bfloat16*>(a.k);
  pp.v = static_cast<const __nv_bfloat16*>(a.v);
  pp.gamma = a.gamma;
  pp.omega = a.omega;
  pp.phi = a.phi;
  pp.H = a.H;
  pp.T = a.T;
  pp.nchunks = nchunks;
  pp.pos0 = a.pos0;
  pp.ws = static_cast<unsigned char*>(a.workspace);
  const unsigned grid = static_cast<unsigned>(bhn) * static_cast<unsigned>(nchunks);
  pow_prep_kernel<6><<<2 * grid, 256, 0, st>>>(pp);
  return cudaGetLastError();
}

cudaError_t pow_fwd_tc_launch(const PowFwdArgs& a, cudaStream_t st) {
  const int bhn = a.B * a.H;
  const int nchunks = (a.T + kC - 1) / kC;
  if (bhn == 0 || nchunks == 0) return cudaSuccess;
  cudaError_t e = pow_set_smem();
  if (e != cudaSuccess) return e;
  PrepParams pp{};
  pp.q = static_cast<const __nv_bfloat16*>(a.q);
  pp.k = static_cast<const __nv_bfloat16*>(a.k);
  pp.v = static_cast<const __nv_bfloat16*>(a.v);
  pp.gamma = a.gamma;
  pp.omega = a.omega;
  pp.phi = a.phi;
  pp.H = a.H;
  pp.T = a.T;
  pp.nchunks = nchunks;
  pp.pos0 = a.pos0;
  pp.ws = static_cast<unsigned char*>(a.workspace);
  const unsigned grid = static_cast<unsigned>(bhn) * static_cast<unsigned>(nchunks);
  pow_prep_kernel<6><<<2 * grid, 256, 0, st>>>(pp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  PowParams p{};
  p.ws = pp.ws;
  p.H = a.H;
  p.T = a.T;
  p.nchunks = nchunks;
  p.bhn = bhn;
  p.eps = a.eps;
  p.o = a.o;
  p.Dn = a.D;
  const ProfileEvents& pe = profile_events();
  const bool rec = pe.start != nullptr;
  if (rec) cudaEventRecord(pe.start, st);
  if (a.p < 1 || a.p > kMaxP) return cudaErrorInvalidValue;
  attn_kernel_for(a.p)<<<grid, kThreads, kSmemBytes, st>>>(p);
  e = cudaGetLastError();
  if (rec) cudaEventRecord(pe.stop, st);
  return e;
}

cudaError_t ablation_fwd_tc_launch(const PowFwdArgs& a, int channels, float shift,
                                  cudaStream_t st) {
  const int bhn = a.B * a.H;
  const int nchunks = (a.T + kC - 1) / kC;
  if (bhn == 0 || nchunks == 0) return cudaSuccess;
  AttnKernel kf = ablation_kernel_for(a.p, channels);
  if (kf == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = pow_set_smem();
  if (e != cudaSuccess) return e;
  PrepParams pp{};
  pp.q = static_cast<const __nv_bfloat16*>(a.q);
  pp.k = static_cast<const __nv_bfloat16*>(a.k);
  pp.v = static_cast<const __nv_bfloat16*>(a.v);
  pp.gamma = a.gamma;
  pp.omega = a.omega;
  pp.phi = a.phi;
  pp.H = a.H;
  pp.T = a.T;
  pp.nchunks = nchunks;
  pp.pos0 = a.pos0;
  pp.ws = static_cast<unsigned char*>(a.workspace);
  const unsigned grid = static_cast<unsigned>(bhn) * static_cast<unsigned>(nchunks);
  if (channels == 4)
    pow_prep_kernel<4><<<2 * grid, 256, 0, st>>>(pp);
  else
    pow_prep_kernel<3><<<2 * grid, 256, 0, st>>>(pp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  PowParams p{};
  p.ws = pp.ws;
  p.H = a.H;
  p.T = a.T;
  p.nchunks = nchunks;
  p.bhn = bhn;
  p.eps = a.eps;
  // score scale: the map's largest score, 3d (four channels) or 2d + shift
  const float c = channels == 4 ? 3.0f * kD : 2.0f * kD + shift;
  p.inv_c = 1.0f / c;
  p.cst = (static_cast<float>(kD) + shift) / c;
  p.o = a.o;
  p.Dn = a.D;
  const ProfileEvents& pe = profile_events();
  const bool rec = pe.start != nullptr;
  if (rec) cudaEventRecord(pe.start, st);
  kf<<<grid, kThreads, kSmemBytes, st>>>(p);
  e = cudaGetLastError();
  if (rec) cudaEventRecord(pe.stop, st);
  return e;
}

int pow_tc_read_and_clear_error(cudaStream_t st) {
  int h = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_pow_tc_error, sizeof(int), 0, cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return -1;
  if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_pow_tc_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                st) != cudaSuccess)
      return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  }
  return h;
}

}  // namespace sanatan
