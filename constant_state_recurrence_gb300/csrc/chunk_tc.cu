// Chunked forward on the tensor cores (tcgen05 + TMEM), bf16 operands with
// f32 accumulation, for sequences of bf16 q, k, v.
//
// The method (reading notes §2.3 and §2.7, paper eqs. (6), (7), (9)):
//   o_t = Phi(q_t)^T S_t / (Phi(q_t)^T z_t + eps),  S_t = sum_{j<=t} Phi(k_j) v_j^T.
// Per chunk of kC = 128 tokens this is evaluated as
//   P      = PhiQ PhiK^T (+ the ones channel, below), masked to j <= t
//   O_ext  = PhiQ [S | z]_prev + P [V | 1]     (columns 0..63: numerator, 64: denominator)
//   [S|z] += PhiK^T [V | 1]
// which is the recurrence re-associated by chunks (the sums are identical).
//
// Feature layout.  Channel 0 of every dimension is the constant 1, so its 64
// features are the same for every token: they contribute exactly 64 to every
// score and 64 * sum(v) to every numerator.  The tensor cores therefore see
// only the 320 non-constant features (c = 1..5 = cos, sin, r, r cos, r sin),
// ordered by groups of eight dimensions, f = 40 (a / 8) + 8 (c - 1) + a % 8;
// the constant channel is added back in the epilogues.  The running sum of v and the token
// count live in an extra state row (row 320) produced by a ones feature of
// PhiK, so they accumulate in f32 on the tensor core with the rest of the
// state.
//
// Roles (768 threads, six warpgroups): warps 0-7 featurise q into Phi(Q) and
// warps 8-15 k into Phi(K) (80 registers each, the launch allocation); warps
// 16-19 drain TMEM (mask + split the scores into bf16 hi/lo parts, snapshot
// the state to bf16 for the next chunk, normalise and store the outputs; 120
// registers after setmaxnreg); one thread of warp 20 issues every
// tcgen05.mma and warps 21-22 copy v rows into shared memory with cp.async
// (that warpgroup keeps 40 registers).  All hand-offs are mbarriers with
// bounded waits.  The next chunk's q, k, v are bulk-prefetched into L2 while
// the current one runs; each output tile is staged in shared memory and
// written with coalesced stores.
//
// Shared-memory operands use the canonical no-swizzle layout (8 x 16-byte
// core matrices); TMEM holds P (128 cols), O_ext (80) and the f32 state
// (3 tiles x 80).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "sanatan_internal.h"
#include "sanatan_math.cuh"
#include "tc_ptx.cuh"
#include "tc_common.cuh"

namespace sanatan {

__device__ int g_tc_error;  // set when a bounded wait gives up

namespace {

using namespace tc;
using namespace tcc;

constexpr uint32_t kTP = 0;          // TMEM columns: P / P-tilde
constexpr uint32_t kTO = 128;        // O_ext
constexpr uint32_t kTS = 208;        // state tiles at 208, 288, 368
constexpr uint32_t kTL = 448;         // low bf16 halves of P-tilde
constexpr uint32_t kTmemCols = 512;

constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + 16 * kXQ;
constexpr int kOffS = kOffK + 16 * kXK;
constexpr int kOffV = kOffS + 40 * kLBO_SV;
// The MMAs read up to 128 B past S'bf16 and V (ignored padding columns); the
// pad keeps those reads inside this layout and away from the mbarriers.
constexpr int kOffMisc = kOffV + 16 * kLBO_SV + 128;
// The state-only pass needs no Phi(Q) and no snapshot: it double-buffers
// Phi(K) and V instead, so that the keys of chunk c + 1 are featurised while
// the tensor core accumulates chunk c.
constexpr int kSoK1 = 16 * kXK;
constexpr int kSoV0 = 2 * 16 * kXK;
constexpr int kSoV1 = kSoV0 + 16 * kLBO_SV;
static_assert(kSoV1 + 16 * kLBO_SV + 128 <= kOffMisc, "state-only buffers must fit");

enum Bar {
  kFeatQ = 0, kFeatK, kFeatV, kPFull, kPTilde, kQFree, kStateDone, kPVDone, kSnapReady, kOFree,
  kDrain,
  // second buffer of Phi(K) / V in the state-only pass
  kFeatK1, kFeatV1, kStateDone1,
  kNumBars
};

struct Misc {
  float4 dimc[64];   // per dim: gamma*sqrt2*cos(omega+pi/4), gamma*sqrt2*sin(omega+pi/4),
                     //          cos(8 phi), sin(8 phi)
  float vs[68];      // state row 320 before the current chunk: sum v (64), count
  float a0[68];      // constant-channel part of S0: sum_a S0[6a] (64), sum_a z0[6a]
  uint64_t bar[kNumBars];
  uint32_t tmem_base;
  int abort_flag;
};
// Output staging: rows at a 272-B (f32) or 144-B (bf16) pitch, so that the
// row-per-thread writes spread over the banks.  It lives in the bf16 state
// snapshot buffer, which is free between the chunk's Phi(Q)[S|z] product and
// the next snapshot.
constexpr int kStagePitch = 272;
constexpr int kStagePitchH = 144;
static_assert(kC * kStagePitch <= 40 * kLBO_SV, "output staging must fit the snapshot buffer");
constexpr int kSmemBytes = kOffMisc + static_cast<int>(sizeof(Misc));
static_assert(kSmemBytes <= 232448, "shared memory layout exceeds 227 KB");

constexpr int kThreads = 768;
// Register split: the block is launched with 768 x 80 registers; the four
// featuriser warpgroups keep 80, the MMA / value-loader warpgroup drops to 40
// and the epilogue warpgroup takes the difference.
constexpr uint32_t kRegLaunch = 80;
constexpr uint32_t kRegEpi = 120;
constexpr uint32_t kRegMma = 40;
static_assert(512 * kRegLaunch + 128 * kRegEpi + 128 * kRegMma <= kThreads * kRegLaunch,
              "setmaxnreg split must fit the launch allocation");
constexpr int kQWarps = 8;     // warps 0-7: query features
constexpr int kKWarp0 = 8;     // warps 8-15: key features
constexpr int kEpiWarp0 = 16;  // warps 16-19: TMEM epilogue
constexpr int kMmaWarp = 20;   // warp 20: MMA issue (one thread)
constexpr int kVWarp0 = 21;    // warps 21-22: value loads
constexpr int kVWarps = 2;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait before giving up

struct TcParams {
  // v as a 4-D tensor {8 columns of a group, token, column group, sequence}
  // (element strides 1, 64, 8, 64 T): one box of 8 x 8 x 8 is the eight 8 x 8
  // core matrices of a token group of [V | 1], in that order (tma_v = 1;
  // forward time only).
  CUtensorMap tmap_v;
  int tma_v;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* gamma;
  const float* omega;
  const float* phi;
  int H, T;
  int64_t pos0;
  float eps;
  int nseg;         // segments per sequence
  int seg_grid;     // CTAs per sequence in this launch
  int nchunks;      // chunks per sequence
  int bhn;          // sequences (B * H); CTA b handles segment b / bhn of sequence b % bhn
  int pdl;          // launched as a programmatic dependent of the state-only pass
  const float* deltas;   // per-segment state sums [B*H][nseg][321][80] (slots 0..nseg-2) or null
  const float* S0;       // full initial state (export of constant rows) or null
  const float* z0;
  float* o;
  float* Dn;
  float* S_out;
  float* z_out;
  float* delta_out;      // state-only mode: compact per-segment sums
  // Modes used by the backward (all off for the forward):
  int reverse;           // process token u as row T-1-u (anti-causal attention)
  int normalize;         // 0: write the numerator N_t instead of N_t / (D_t + eps)
  int out_bf16;          // write o as bf16 instead of f32
  const float* extra;    // per-token value of the ones column of [V | 1] (null: 1)
};

// Row of the sequence that processing position u stands for.
__device__ __forceinline__ int orow(const TcParams& prm, int u) {
  return prm.reverse ? prm.T - 1 - u : u;
}

__device__ __forceinline__ bool wait_bar(Misc& m, int b, uint32_t parity) {
  if (*reinterpret_cast<volatile int*>(&m.abort_flag)) return false;
  if (mbar_wait_bounded(&m.bar[b], parity, kWaitNs)) return true;
  m.abort_flag = 1;
  atomicOr(&g_tc_error, 1);
  return false;
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// L2 prefetch of one chunk's rows of q (unless state-only), k and v.
template <bool kStateOnly>
__device__ __forceinline__ void prefetch_chunk(const TcParams& prm, int64_t seq_row0, int chunk) {
  const int tok0 = chunk * kC;
  const int n = min(kC, prm.T - tok0);
  if (n <= 0) return;
  const int64_t off = (seq_row0 + (prm.reverse ? prm.T - tok0 - n : tok0)) * kD;
  const uint32_t bytes = static_cast<uint32_t>(n) * kD * 2;
  if (!kStateOnly) prefetch_l2_bulk(prm.q + off, bytes);
  prefetch_l2_bulk(prm.k + off, bytes);
  prefetch_l2_bulk(prm.v + off, bytes);
}

// ---------------------------------------------------------------------------
template <bool kStateOnly>
__global__ void __launch_bounds__(kThreads, 1) sanatan_tc_kernel(const __grid_constant__ TcParams prm) {
  extern __shared__ __align__(1024) unsigned char smem[];
  Misc& m = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const uint32_t sQ = smem_u32(smem + kOffQ);
  const uint32_t sK = smem_u32(smem + kOffK);
  const uint32_t sS = smem_u32(smem + kOffS);
  const uint32_t sV = smem_u32(smem + kOffV);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // Segment-major CTA order: the first segments' CTAs are scheduled first (in
  // a dependent launch they need nothing from the state-only pass).
  const int seg = blockIdx.x / prm.bhn;
  const int bh = blockIdx.x % prm.bhn;
  const int h = bh % prm.H;
  const int c_begin = seg_begin(seg, prm.nchunks, prm.nseg);
  const int c_end = seg_begin(seg + 1, prm.nchunks, prm.nseg);
  const int nloc = c_end - c_begin;
  const int64_t seq_row0 = static_cast<int64_t>(bh) * prm.T;  // first token row of the sequence
  const bool last_seg = (seg == prm.nseg - 1);

  // The main pass may be launched (and start its first segments) while this
  // state-only pass runs; it waits for its completion before reading the sums.
  if constexpr (kStateOnly) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    if (nloc > 0) prefetch_chunk<kStateOnly>(prm, seq_row0, c_begin);
    if (nloc > 1) prefetch_chunk<kStateOnly>(prm, seq_row0, c_begin + 1);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&m.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b) {
      // In the state-only pass both featuriser groups produce keys.
      const uint32_t cnt = (b == kFeatQ) ? kQWarps
                           : (b == kFeatK || b == kFeatK1) ? (kStateOnly ? 16u : 8u)
                           : (b == kFeatV || b == kFeatV1) ? static_cast<uint32_t>(kVWarps)
                           : (b == kPTilde || b == kSnapReady || b == kOFree) ? 4u : 1u;
      mbar_init(&m.bar[b], cnt);
    }
    m.abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < kD) {
    const float g = prm.gamma[h] * 1.41421356237309515f;
    float sw, cw;
    sincosf(prm.omega[h * kD + tid] + 0.785398163397448310f, &sw, &cw);
    float s8, c8;
    sincosf(phase_mod_2pi(8, prm.phi[h * kD + tid]), &s8, &c8);
    // In reverse mode consecutive processing positions step back by one row.
    m.dimc[tid] = make_float4(g * cw, g * sw, c8, prm.reverse ? -s8 : s8);
  }
  if (tid >= 64 && tid < 64 + 68) {
    const int e = tid - 64;
    float acc = 0.f;
    if (prm.S0 != nullptr && e < 64) {
      const float* s0 = prm.S0 + static_cast<int64_t>(bh) * 384 * 64;
      for (int a = 0; a < kD; ++a) acc += s0[(6 * a) * 64 + e];
    } else if (prm.z0 != nullptr && e == 64) {
      const float* z0 = prm.z0 + static_cast<int64_t>(bh) * 384;
      for (int a = 0; a < kD; ++a) acc += z0[6 * a];
    }
    m.a0[e] = acc;
  }
  // Constant part of [V | 1 | 0]: column 64 is one, 65..71 zero.
  if (tid < 16 * 8) {
    const int kg = tid >> 3, row = tid & 7;
    if constexpr (kStateOnly) {
      st_shared_v4(smem_u32(smem + kSoV0) + kg * kLBO_SV + 8 * 128 + row * 16, 0x3F80u, 0u, 0u, 0u);
      st_shared_v4(smem_u32(smem + kSoV1) + kg * kLBO_SV + 8 * 128 + row * 16, 0x3F80u, 0u, 0u, 0u);
    } else {
      st_shared_v4(sV + kg * kLBO_SV + 8 * 128 + row * 16, 0x3F80u, 0u, 0u, 0u);
    }
  }
  if (tid < 8) st_shared_v4(sV + 16 * kLBO_SV + 16 * tid, 0u, 0u, 0u, 0u);  // over-read pad
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ featurisers
    // Warps 0-7 write Phi(Q), warps 8-15 Phi(K) (in the state-only pass both
    // groups write Phi(K), two tokens each).  Lane (r, dimension group ag)
    // owns tokens tq + 8 i of the chunk.  The block keeps its launch registers.
    const bool kgrp = kStateOnly || warp >= kKWarp0;
    const int fw = warp & 7;
    const int r = lane & 7;
    const int ag = (lane >> 3) + 4 * (fw & 1);
    constexpr int kNI = kStateOnly ? 2 : 4;  // tokens per thread
    const int tq = 32 * (fw >> 1) + r + ((kStateOnly && warp < kKWarp0) ? 16 : 0);
    const float4* dimc = &m.dimc[8 * ag];
    const float* phi_g = prm.phi + h * kD + 8 * ag;
    const __nv_bfloat16* src = kgrp ? prm.k : prm.q;
    const uint32_t sdst0 = kgrp ? sK : sQ;
    const int pitch = kgrp ? kXK : kXQ;
    // Raw rows of chunk `chunk` for this thread's tokens (zero past the end).
    // They are loaded right after a hand-off and consumed after the next wait:
    // an mbarrier arrive has release semantics and would stall on loads still
    // in flight.
    uint4 raw[kNI];
    auto load_raw = [&](int chunk) {
      const int tok0 = chunk * kC;
#pragma unroll
      for (int i = 0; i < kNI; ++i) {
        const int t = tq + 8 * i;
        raw[i] = (chunk < c_end && tok0 + t < prm.T)
                     ? ldg_nc_v4(src + (seq_row0 + orow(prm, tok0 + t)) * kD + 8 * ag)
                     : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    load_raw(c_begin);
    for (int ci = 0; ci < nloc; ++ci) {
      const int chunk = c_begin + ci;
      const int tok0 = chunk * kC;
      if (tid == 0 && ci + 2 < nloc) prefetch_chunk<kStateOnly>(prm, seq_row0, chunk + 2);
      float cb[8], sb[8];
      {
        const int64_t tabs = prm.pos0 + orow(prm, tok0 + tq);
#pragma unroll
        for (int j = 0; j < 8; ++j) __sincosf(phase_mod_2pi(tabs, __ldg(phi_g + j)), &sb[j], &cb[j]);
      }
      // The buffer is free once the MMAs of its previous chunk have read it.
      uint32_t sdst = sdst0;
      if constexpr (kStateOnly) {
        sdst = smem_u32(smem) + (ci & 1) * kSoK1;
        if (ci > 1) wait_bar(m, (ci & 1) ? kStateDone1 : kStateDone, ((ci >> 1) - 1) & 1);
      } else {
        if (ci > 0) wait_bar(m, kgrp ? kStateDone : kQFree, (ci - 1) & 1);
      }
#pragma unroll
      for (int i = 0; i < kNI; ++i) {
        const int t = tq + 8 * i;
        const bool valid = tok0 + t < prm.T;
        uint32_t f[5][4];
        if (valid) {
          features8(raw[i], dimc, cb, sb, f);
        } else {
#pragma unroll
          for (int c = 0; c < 5; ++c)
#pragma unroll
            for (int p = 0; p < 4; ++p) f[c][p] = 0u;
        }
        const uint32_t base = sdst + (t >> 3) * pitch + (t & 7) * 16;
#pragma unroll
        for (int c = 0; c < 5; ++c)
          st_shared_v4(base + feat_group(ag, c + 1) * 128, f[c][0], f[c][1], f[c][2], f[c][3]);
        if (kgrp && ag == 0) st_shared_v4(base + 40 * 128, valid ? 0x3F80u : 0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 kc = dimc[j];
          const float nc = fmaf(cb[j], kc.z, -sb[j] * kc.w);
          sb[j] = fmaf(sb[j], kc.z, cb[j] * kc.w);
          cb[j] = nc;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0)
        mbar_arrive(&m.bar[kStateOnly ? ((ci & 1) ? kFeatK1 : kFeatK) : (kgrp ? kFeatK : kFeatQ)]);
      load_raw(chunk + 1);
    }
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------------ TMEM epilogue
    setmaxnreg_inc<kRegEpi>();
    const int qd = warp - kEpiWarp0;           // TMEM lane quarter
    const int row = 32 * qd + lane;            // TMEM lane = token row / feature row in tile
    const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
    // Initial state -> TMEM tiles (and the bf16 snapshot for the first chunk):
    // the caller's state (S0, z0) plus the sums of all earlier segments.
    if (!kStateOnly && prm.pdl && seg > 0)
      asm volatile("griddepcontrol.wait;" ::: "memory");  // the state-only pass is complete
    {
      for (int mt = 0; mt < 3; ++mt) {
        const int f = mt * 128 + row;
        if (mt == 2 && qd == 3) continue;  // rows 352..383 are never used
        float val[80];
#pragma unroll
        for (int e = 0; e < 80; ++e) val[e] = 0.f;
        if (!kStateOnly && f < kNF && prm.S0 != nullptr) {
          int a, c;
          feat_dim_chan(f, a, c);
          const int64_t rowi = static_cast<int64_t>(bh) * 384 + 6 * a + c;
          const float4* s4 = reinterpret_cast<const float4*>(prm.S0 + rowi * 64);
#pragma unroll
          for (int e4 = 0; e4 < 16; ++e4) {
            const float4 x = s4[e4];
            val[4 * e4] = x.x; val[4 * e4 + 1] = x.y; val[4 * e4 + 2] = x.z; val[4 * e4 + 3] = x.w;
          }
          val[64] = prm.z0[rowi];
        }
        if (!kStateOnly && f < kSCRows && prm.deltas != nullptr) {
          const float* d0 = prm.deltas + static_cast<int64_t>(bh) * prm.nseg * kSCRows * kSCCols;
          for (int sp = 0; sp < seg; ++sp) {
            const float* ds = d0 + static_cast<int64_t>(sp) * kSCRows * kSCCols;
#pragma unroll
            for (int e = 0; e < 65; ++e) val[e] += ds[sc_index(f, e)];
          }
        }
#pragma unroll
        for (int blk = 0; blk < 5; ++blk) {
          uint32_t rr[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) rr[i] = __float_as_uint(val[16 * blk + i]);
          tmem_st16(tmem + lane_off + kTS + mt * kN + 16 * blk, rr);
        }
        if constexpr (!kStateOnly) {
          if (f < kNF) {
            const uint32_t base = sS + (f >> 3) * kLBO_SV + (f & 7) * 16;
#pragma unroll
            for (int ng = 0; ng < kNG; ++ng)
              st_shared_v4(base + ng * 128, pack_bf16x2(val[8 * ng], val[8 * ng + 1]),
                           pack_bf16x2(val[8 * ng + 2], val[8 * ng + 3]),
                           pack_bf16x2(val[8 * ng + 4], val[8 * ng + 5]),
                           pack_bf16x2(val[8 * ng + 6], val[8 * ng + 7]));
          } else if (f == kNF) {
#pragma unroll
            for (int e = 0; e < 65; ++e) m.vs[e] = val[e];
          }
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      epi_sync();
      if (lane == 0) {
        mbar_arrive(&m.bar[kSnapReady]);
        mbar_arrive(&m.bar[kOFree]);
      }
    }
    if constexpr (!kStateOnly) {
      for (int ci = 0; ci < nloc; ++ci) {
        const int tok0 = (c_begin + ci) * kC;
        // E1: mask the scores, add the constant channel, split into bf16 hi + lo.
        // Keys are taken 32 at a time; the hi halves overwrite P in place (their
        // columns hold keys that were already read), the lo halves go to kTL.
        wait_bar(m, kPFull, ci & 1);
        tc_fence_after();
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t hi[16], lo[16];
          if (b > qd) {  // every key of this block is after every row of this warp
#pragma unroll
            for (int i = 0; i < 16; ++i) { hi[i] = 0u; lo[i] = 0u; }
          } else {
            float p[32];
            tmem_ld16(tmem + lane_off + kTP + 32 * b, *reinterpret_cast<float(*)[16]>(&p[0]));
            tmem_ld16(tmem + lane_off + kTP + 32 * b + 16, *reinterpret_cast<float(*)[16]>(&p[16]));
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j0 = 32 * b + 2 * i;
              const float x0 = (j0 <= row) ? p[2 * i] + 64.0f : 0.0f;
              const float x1 = (j0 + 1 <= row) ? p[2 * i + 1] + 64.0f : 0.0f;
              const uint32_t hpk = pack_bf16x2(x0, x1);
              hi[i] = hpk;
              lo[i] = pack_bf16x2(x0 - __uint_as_float(hpk << 16),
                                  x1 - __uint_as_float(hpk & 0xffff0000u));
            }
          }
          tmem_st16(tmem + lane_off + kTP + 16 * b, hi);
          tmem_st16(tmem + lane_off + kTL + 16 * b, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&m.bar[kPTilde]);

        // E3: outputs of this chunk (state row 320 in m.vs is still the pre-chunk one).
        // Each row is normalised in registers and staged in the free snapshot
        // buffer; the four warps then copy the staged tile out with coalesced
        // 16-byte stores (each warp instruction writes whole rows).
        wait_bar(m, kPVDone, ci & 1);
        tc_fence_after();
        const int nrow = min(kC, prm.T - tok0);
        {
          float ov[80];
#pragma unroll
          for (int blk = 0; blk < 5; ++blk) {
            float x[16];
            tmem_ld16(tmem + lane_off + kTO + 16 * blk, x);
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[16 * blk + i] = x[i];
          }
          tmem_ld_wait();
          if (row < nrow) {
            const float den = ov[64] + 64.0f * m.vs[64] + m.a0[64];
            const float inv = prm.normalize ? 1.0f / (den + prm.eps) : 1.0f;
            const float4* vs4 = reinterpret_cast<const float4*>(m.vs);
            const float4* a04 = reinterpret_cast<const float4*>(m.a0);
#pragma unroll
            for (int e4 = 0; e4 < 16; ++e4) {
              const float4 w = vs4[e4];
              const float4 c = a04[e4];
              ov[4 * e4 + 0] = (fmaf(64.0f, w.x, ov[4 * e4 + 0]) + c.x) * inv;
              ov[4 * e4 + 1] = (fmaf(64.0f, w.y, ov[4 * e4 + 1]) + c.y) * inv;
              ov[4 * e4 + 2] = (fmaf(64.0f, w.z, ov[4 * e4 + 2]) + c.z) * inv;
              ov[4 * e4 + 3] = (fmaf(64.0f, w.w, ov[4 * e4 + 3]) + c.w) * inv;
            }
            if (prm.out_bf16) {
              const uint32_t srow = sS + row * kStagePitchH;
#pragma unroll
              for (int e8 = 0; e8 < 8; ++e8)
                st_shared_v4(srow + 16 * e8, pack_bf16x2(ov[8 * e8], ov[8 * e8 + 1]),
                             pack_bf16x2(ov[8 * e8 + 2], ov[8 * e8 + 3]),
                             pack_bf16x2(ov[8 * e8 + 4], ov[8 * e8 + 5]),
                             pack_bf16x2(ov[8 * e8 + 6], ov[8 * e8 + 7]));
            } else {
              const uint32_t srow = sS + row * kStagePitch;
#pragma unroll
              for (int e4 = 0; e4 < 16; ++e4)
                st_shared_v4(srow + 16 * e4, __float_as_uint(ov[4 * e4]),
                             __float_as_uint(ov[4 * e4 + 1]), __float_as_uint(ov[4 * e4 + 2]),
                             __float_as_uint(ov[4 * e4 + 3]));
            }
            if (prm.Dn != nullptr) prm.Dn[seq_row0 + orow(prm, tok0 + row)] = den;
          }
        }
        tc_fence_before();
        epi_sync();  // every row staged, every thread done with m.vs and O
        if (lane == 0) mbar_arrive(&m.bar[kOFree]);
        {
          // 16-byte pieces: piece p is column piece p % per_row of staged row p / per_row.
          const int et = tid - 32 * kEpiWarp0;
          const int lg = prm.out_bf16 ? 3 : 4;  // log2 of pieces per row
          const int pitch = prm.out_bf16 ? kStagePitchH : kStagePitch;
          unsigned char* obase = reinterpret_cast<unsigned char*>(prm.o);
          const int64_t row_bytes = int64_t{16} << lg;
          for (int pc = et; pc < (nrow << lg); pc += 128) {
            const int rr = pc >> lg, cc = pc & ((1 << lg) - 1);
            const uint4 val = *reinterpret_cast<const uint4*>(smem + kOffS + rr * pitch + 16 * cc);
            *reinterpret_cast<uint4*>(obase + (seq_row0 + orow(prm, tok0 + rr)) * row_bytes +
                                      16 * cc) = val;
          }
        }
        epi_sync();  // staged tile read out before the snapshot overwrites it

        // E2: snapshot of the state after this chunk, for the next chunk.
        wait_bar(m, kStateDone, ci & 1);
        tc_fence_after();
        if (ci + 1 < nloc) {
          for (int mt = 0; mt < 3; ++mt) {
            if (mt == 2 && qd >= 3) continue;
            const int f = mt * 128 + row;
            float val[72];
#pragma unroll
            for (int blk = 0; blk < 5; ++blk) {
              float x[16];
              tmem_ld16(tmem + lane_off + kTS + mt * kN + 16 * blk, x);
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (16 * blk + i < 72) val[16 * blk + i] = x[i];
            }
            tmem_ld_wait();
            if (f < kNF) {
              const uint32_t base = sS + (f >> 3) * kLBO_SV + (f & 7) * 16;
#pragma unroll
              for (int ng = 0; ng < kNG; ++ng)
                st_shared_v4(base + ng * 128, pack_bf16x2(val[8 * ng], val[8 * ng + 1]),
                             pack_bf16x2(val[8 * ng + 2], val[8 * ng + 3]),
                             pack_bf16x2(val[8 * ng + 4], val[8 * ng + 5]),
                             pack_bf16x2(val[8 * ng + 6], val[8 * ng + 7]));
            } else if (f == kNF) {
#pragma unroll
              for (int e = 0; e < 65; ++e) m.vs[e] = val[e];
            }
          }
          fence_proxy_async_smem();
          tc_fence_before();
          epi_sync();
          if (lane == 0) mbar_arrive(&m.bar[kSnapReady]);
        }
      }
    } else {
      // One wait on the single-phase drain barrier: a wait on the last
      // state_done phase could alias an earlier phase of the same parity.
      wait_bar(m, kDrain, 0);
      tc_fence_after();
    }
    // Final state of the segment: the sequence's S_out / z_out (last segment of
    // a full pass) or the per-segment sums (state-only pass).
    const bool want_export = kStateOnly ? (prm.delta_out != nullptr)
                                        : (last_seg && prm.S_out != nullptr);
    if (want_export) {
      for (int mt = 0; mt < 3; ++mt) {
        if (mt == 2 && qd >= 3) continue;
        const int f = mt * 128 + row;
        float val[80];
#pragma unroll
        for (int blk = 0; blk < 5; ++blk) {
          float x[16];
          tmem_ld16(tmem + lane_off + kTS + mt * kN + 16 * blk, x);
#pragma unroll
          for (int i = 0; i < 16; ++i) val[16 * blk + i] = x[i];
        }
        tmem_ld_wait();
        if (kStateOnly) {
          if (f < kSCRows) {
            float* dst = prm.delta_out + (static_cast<int64_t>(bh) * prm.nseg + seg) * kSCRows * kSCCols;
#pragma unroll
            for (int e = 0; e < 65; ++e) dst[sc_index(f, e)] = val[e];
          }
        } else {
          if (f < kNF) {
            int a, c;
            feat_dim_chan(f, a, c);
            float4* dst = reinterpret_cast<float4*>(prm.S_out + (static_cast<int64_t>(bh) * 384 +
                                                                 6 * a + c) * 64);
#pragma unroll
            for (int e4 = 0; e4 < 16; ++e4)
              dst[e4] = make_float4(val[4 * e4], val[4 * e4 + 1], val[4 * e4 + 2], val[4 * e4 + 3]);
            prm.z_out[static_cast<int64_t>(bh) * 384 + 6 * a + c] = val[64];
          } else if (f == kNF) {
#pragma unroll
            for (int e = 0; e < 65; ++e) m.vs[e] = val[e];
          }
        }
      }
      if (!kStateOnly) {
        epi_sync();
        // constant-channel rows: S0[6a] + sum v, z0[6a] + count
        const int et = tid - 32 * kEpiWarp0;
        for (int idx = et; idx < kD * 65; idx += 128) {
          const int a = idx / 65, e = idx % 65;
          const int64_t rowi = static_cast<int64_t>(bh) * 384 + 6 * a;
          if (e < 64) {
            const float base = prm.S0 ? prm.S0[rowi * 64 + e] : 0.f;
            prm.S_out[rowi * 64 + e] = base + m.vs[e];
          } else {
            const float base = prm.z0 ? prm.z0[rowi] : 0.f;
            prm.z_out[rowi] = base + m.vs[64];
          }
        }
      }
    }
  } else {
    setmaxnreg_dec<kRegMma>();
  }
  if (warp >= kVWarp0 && warp < kVWarp0 + kVWarps) {
    // ------------------------------------------------------------ value loads
    // v rows go straight to [V | 1] in shared memory, by TMA tensor copies in
    // forward time and 16-byte cp.async copies otherwise (the ones column is
    // constant; the optional extra column replaces it per token).
    const int vt = tid - 32 * kVWarp0;
    int tma_issued = 0;   // chunks whose tensor copies have been issued
    for (int ci = 0; ci < nloc; ++ci) {
      const int tok0 = (c_begin + ci) * kC;
      const int nrow = min(kC, prm.T - tok0);
      uint32_t vdst = sV;
      uint64_t* vbar = &m.bar[(kStateOnly && (ci & 1)) ? kFeatV1 : kFeatV];
      bool free_buf = true;
      if constexpr (kStateOnly) {
        vdst = smem_u32(smem + ((ci & 1) ? kSoV1 : kSoV0));
        if (ci > 1) free_buf = wait_bar(m, (ci & 1) ? kStateDone1 : kStateDone, ((ci >> 1) - 1) & 1);
      } else {
        if (ci > 0) free_buf = wait_bar(m, kPVDone, (ci - 1) & 1);
      }
      // after an abandoned wait no further asynchronous copy is issued
      if (!free_buf && prm.tma_v) break;
      if (prm.tma_v) {
        // 16 tensor loads of one token group each (rows past the end read as
        // zero); the first value-loader thread's arrival carries their bytes
        if (vt == 0) {
          mbar_arrive_expect_tx(vbar, 16u * 8u * 128u);
          for (int kg = 0; kg < 16; ++kg)
            tma_load_4d(vdst + kg * kLBO_SV, &prm.tmap_v, 0, tok0 + 8 * kg, 0, bh, vbar);
        }
        tma_issued = ci + 1;
        if (prm.extra != nullptr) {
          for (int t = vt; t < kC; t += 32 * kVWarps) {
            const float x = t < nrow ? prm.extra[seq_row0 + orow(prm, tok0 + t)] : 0.f;
            st_shared_v4(vdst + (t >> 3) * kLBO_SV + 8 * 128 + (t & 7) * 16,
                         __bfloat16_as_ushort(__float2bfloat16_rn(x)), 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && vt != 0) mbar_arrive(vbar);
        continue;
      }
      for (int pc = vt; pc < kC * 8; pc += 32 * kVWarps) {
        const int t = pc >> 3, ng = pc & 7;
        const bool valid = t < nrow;
        const __nv_bfloat16* gsrc =
            prm.v + (seq_row0 + orow(prm, tok0 + (valid ? t : 0))) * kD + 8 * ng;
        cp_async_16(vdst + (t >> 3) * kLBO_SV + ng * 128 + (t & 7) * 16, gsrc, valid ? 16u : 0u);
      }
      if (prm.extra != nullptr) {
        for (int t = vt; t < kC; t += 32 * kVWarps) {
          const float x = t < nrow ? prm.extra[seq_row0 + orow(prm, tok0 + t)] : 0.f;
          st_shared_v4(vdst + (t >> 3) * kLBO_SV + 8 * 128 + (t & 7) * 16,
                       __bfloat16_as_ushort(__float2bfloat16_rn(x)), 0u, 0u, 0u);
        }
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&m.bar[(kStateOnly && (ci & 1)) ? kFeatV1 : kFeatV]);
    }
    // No tensor copy may still be writing shared memory when the CTA exits,
    // also after an abandoned wait: wait (bounded) for the last issued ones.
    if (vt == 0) {
      for (int ci = (tma_issued >= 2 ? tma_issued - 2 : 0); ci < tma_issued; ++ci) {
        if (kStateOnly)
          mbar_wait_bounded(&m.bar[(ci & 1) ? kFeatV1 : kFeatV], (ci >> 1) & 1, kWaitNs);
        else if (ci == tma_issued - 1)
          mbar_wait_bounded(&m.bar[kFeatV], ci & 1, kWaitNs);
      }
    }
  }
  if (warp == kMmaWarp && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idQK = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idIN = idesc_bf16_f32(128, kN, false, true);
    constexpr uint32_t idST = idesc_bf16_f32(128, kN, true, true);
    constexpr uint32_t idPV = idesc_bf16_f32(128, kN, false, true);
    // Descriptor bases; an operand at byte offset o from its base is base + o/16
    // (the start-address field is the low 14 bits and never overflows here).
    // The issue stream is fully unrolled: a rolled loop costs the single
    // issuing thread more cycles per MMA than the tensor core needs.
    const uint64_t dQ = smem_desc(sQ, 128, kXQ);          // PhiQ, K-major A
    const uint64_t dKb = smem_desc(sK, 128, kXK);         // PhiK, K-major B (scores)
    const uint64_t dKa = smem_desc(sK, kXK, 128);         // PhiK^T, MN-major A (state)
    const uint64_t dS = smem_desc(sS, kLBO_SV, 128);      // S' bf16, MN-major B
    const uint64_t dV = smem_desc(sV, kLBO_SV, 128);      // [V | 1], MN-major B
    for (int ci = 0; ci < nloc; ++ci) {
      // Opaque copies of the bases keep the descriptor arithmetic of each group
      // next to its MMAs instead of hoisted (80 live descriptors would not fit
      // this warpgroup's registers).
      uint64_t dQl = dQ, dKbl = dKb, dKal = dKa, dSl = dS, dVl = dV;
      if constexpr (kStateOnly) {
        // double-buffered Phi(K) and V: chunk ci uses buffer ci & 1
        dKal = smem_desc(smem_u32(smem) + (ci & 1) * kSoK1, kXK, 128);
        dVl = smem_desc(smem_u32(smem + ((ci & 1) ? kSoV1 : kSoV0)), kLBO_SV, 128);
      }
      asm volatile("" : "+l"(dQl), "+l"(dKbl), "+l"(dKal), "+l"(dSl), "+l"(dVl));
      if constexpr (kStateOnly) {
        wait_bar(m, (ci & 1) ? kFeatK1 : kFeatK, (ci >> 1) & 1);
      } else {
        wait_bar(m, kFeatQ, ci & 1);
        wait_bar(m, kFeatK, ci & 1);
      }
      tc_fence_after();
      if constexpr (!kStateOnly) {
#pragma unroll
        for (int s = 0; s < 20; ++s)
          mma_ss(tmem + kTP, dQl + 16 * s, dKbl + 16 * s, idQK, s > 0);
        mma_commit(&m.bar[kPFull]);
        wait_bar(m, kSnapReady, ci & 1);  // bf16 state snapshot of the previous chunk
        wait_bar(m, kOFree, ci & 1);      // previous outputs drained from TMEM
        tc_fence_after();
        asm volatile("" : "+l"(dQl), "+l"(dSl));
#pragma unroll
        for (int s = 0; s < 20; ++s)
          mma_ss(tmem + kTO, dQl + 16 * s, dSl + (2 * kLBO_SV / 16) * s, idIN, s > 0);
        mma_commit(&m.bar[kQFree]);
      } else if (ci == 0) {
        wait_bar(m, kSnapReady, 0);  // initial state is in TMEM
        tc_fence_after();
      }
      if constexpr (kStateOnly)
        wait_bar(m, (ci & 1) ? kFeatV1 : kFeatV, (ci >> 1) & 1);
      else
        wait_bar(m, kFeatV, ci & 1);
      tc_fence_after();
      asm volatile("" : "+l"(dKal), "+l"(dVl));
#pragma unroll
      for (int s = 0; s < 8; ++s)
#pragma unroll
        for (int mt = 0; mt < 3; ++mt)
          mma_ss(tmem + kTS + mt * kN, dKal + (2048 / 16) * mt + (2 * kXK / 16) * s,
                 dVl + (2 * kLBO_SV / 16) * s, idST, true);
      mma_commit(&m.bar[(kStateOnly && (ci & 1)) ? kStateDone1 : kStateDone]);
      if constexpr (!kStateOnly) {
        wait_bar(m, kPTilde, ci & 1);
        tc_fence_after();
        asm volatile("" : "+l"(dVl));
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint64_t bd = dVl + (2 * kLBO_SV / 16) * s;
          mma_ts(tmem + kTO, tmem + kTP + 8 * s, bd, idPV, true);
          mma_ts(tmem + kTO, tmem + kTL + 8 * s, bd, idPV, true);
        }
      }
      mma_commit(&m.bar[kPVDone]);
    }
    // Nothing may still be in flight when TMEM is released: wait (bounded) for
    // the drain even after an abandoned wait, when wait_bar returns at once.
    mma_commit(&m.bar[kDrain]);
    mbar_wait_bounded(&m.bar[kDrain], 0, kWaitNs);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int sm_count() {
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

}  // namespace

int tc_segments(int B, int H, int T) {
  const int64_t bhn = static_cast<int64_t>(B) * H;
  const int nchunks = (T + kC - 1) / kC;
  if (bhn <= 0 || nchunks <= 1) return 1;
  const int64_t sms = sm_count();
  const int64_t per = sms / bhn;
  if (per <= 1) {
    if (bhn >= sms) return 1;
    // With about one CTA per sequence some SMs would idle.  More segments run
    // as several waves of one-CTA-per-SM work: pick the count that minimises
    // waves x chunks per segment, charging one chunk for the state-only pass
    // that any split needs.
    int best = 1;
    int64_t best_cost = (bhn + sms - 1) / sms * nchunks;
    for (int sg = 2; sg <= 8 && sg <= nchunks; ++sg) {
      const int64_t waves = (bhn * sg + sms - 1) / sms;
      const int64_t cost = waves * ((nchunks + sg - 1) / sg) + 1;
      if (cost < best_cost) { best_cost = cost; best = sg; }
    }
    return best;
  }
  return static_cast<int>(per < nchunks ? per : nchunks);
}

int tc_segments_fit(int B, int H, int T, size_t bytes) {
  const size_t slot = static_cast<size_t>(B) * H * kSCRows * kSCCols * sizeof(float);
  int sg = tc_segments(B, H, T);
  while (sg > 1 && static_cast<size_t>(sg) * slot > bytes) --sg;
  return sg;
}

size_t chunk_fwd_tc_workspace_bytes(int B, int H, int T) {
  const int nseg = tc_segments(B, H, T);
  if (nseg <= 1) return 0;  // one segment reads and writes no per-segment sums
  return static_cast<size_t>(B) * H * nseg * kSCRows * kSCCols * sizeof(float);
}

namespace {

// The shared-memory opt-in is a per-device attribute of the kernel: set it once.
cudaError_t tc_set_smem() {
  static bool done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(sanatan_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(sanatan_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

// cuTensorMapEncodeTiled, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// The tensor map of v for the value loads (see TcParams::tmap_v); false when
// it cannot be encoded (the loads then use cp.async).
bool encode_value_map(CUtensorMap* map, const void* v, int bhn, int T) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {8, static_cast<cuuint64_t>(T), 8, static_cast<cuuint64_t>(bhn)};
  const cuuint64_t strides[3] = {kD * 2, 16, static_cast<cuuint64_t>(T) * kD * 2};
  const cuuint32_t box[4] = {8, 8, 8, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(v), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

TcParams tc_params(const TcJob& job) {
  TcParams p{};
  // value loads by tensor copies in forward time (the reversed rows of the
  // backward's passes keep the row-by-row copies)
  if (!job.reverse && job.T > 0 && job.B * job.H > 0)
    p.tma_v = encode_value_map(&p.tmap_v, job.v, job.B * job.H, job.T) ? 1 : 0;
  p.q = static_cast<const __nv_bfloat16*>(job.q);
  p.k = static_cast<const __nv_bfloat16*>(job.k);
  p.v = static_cast<const __nv_bfloat16*>(job.v);
  p.gamma = job.gamma;
  p.omega = job.omega;
  p.phi = job.phi;
  p.H = job.H;
  p.T = job.T;
  p.pos0 = job.pos0;
  p.eps = job.eps;
  p.nseg = job.nseg > 0 ? job.nseg : tc_segments(job.B, job.H, job.T);
  p.bhn = job.B * job.H;
  p.nchunks = (job.T + kC - 1) / kC;
  p.reverse = job.reverse;
  p.normalize = job.normalize;
  p.out_bf16 = job.out_bf16;
  p.extra = job.extra;
  return p;
}

}  // namespace

cudaError_t tc_state_pass(const TcJob& job, cudaStream_t st) {
  cudaError_t e = tc_set_smem();
  if (e != cudaSuccess) return e;
  TcParams d = tc_params(job);
  if (d.nseg <= 1) return cudaSuccess;
  // The sum of each segment but the last -> deltas[bh][p].  A main pass then
  // starts segment p from S0 plus the sums of segments < p.
  d.seg_grid = d.nseg - 1;
  d.delta_out = job.deltas;
  sanatan_tc_kernel<true><<<job.B * job.H * (d.nseg - 1), kThreads, kSmemBytes, st>>>(d);
  return cudaGetLastError();
}

cudaError_t tc_attention(const TcJob& job, cudaStream_t st) {
  cudaError_t e = tc_set_smem();
  if (e != cudaSuccess) return e;
  TcParams p = tc_params(job);
  const bool state_pass = p.nseg > 1 && !job.deltas_ready;
  if (state_pass) {
    if ((e = tc_state_pass(job, st)) != cudaSuccess) return e;
  }
  p.seg_grid = p.nseg;
  p.deltas = p.nseg > 1 ? job.deltas : nullptr;
  p.S0 = job.S0;
  p.z0 = job.z0;
  p.o = static_cast<float*>(job.o);
  p.Dn = job.Dn;
  p.S_out = job.S_out;
  p.z_out = job.z_out;
  const ProfileEvents& pe = profile_events();
  const bool rec = job.record_events && pe.start != nullptr;
  if (rec) cudaEventRecord(pe.start, st);
  const unsigned grid = static_cast<unsigned>(job.B * job.H * p.nseg);
  if (state_pass && !rec) {
    // Programmatic dependent launch: the main pass starts as soon as SMs free
    // up; only CTAs of segments > 0 wait for the state-only pass.
    p.pdl = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, sanatan_tc_kernel<false>, p);
  } else {
    sanatan_tc_kernel<false><<<grid, kThreads, kSmemBytes, st>>>(p);
    e = cudaGetLastError();
  }
  if (rec) cudaEventRecord(pe.stop, st);
  return e;
}

cudaError_t chunk_fwd_tc_launch(const ChunkFwdArgs& a, cudaStream_t st) {
  TcJob job;
  job.q = a.q;
  job.k = a.k;
  job.v = a.v;
  job.gamma = a.gamma;
  job.omega = a.omega;
  job.phi = a.phi;
  job.B = a.B;
  job.H = a.H;
  job.T = a.T;
  job.pos0 = a.pos0;
  job.eps = a.eps;
  job.S0 = a.S0;
  job.z0 = a.z0;
  job.o = a.o;
  job.Dn = a.D;
  job.S_out = a.S_out;
  job.z_out = a.z_out;
  job.deltas = static_cast<float*>(a.workspace);
  job.nseg = tc_segments_fit(a.B, a.H, a.T, a.workspace_bytes);
  return tc_attention(job, st);
}

namespace {
// Failure-detection probe: one thread waits, with the kernels' bounded wait,
// on an mbarrier that nothing arrives at (unless `arrive`), and records a
// timeout in the same error word as the tensor-core kernels.
__global__ void timeout_probe_kernel(uint64_t timeout_ns, int arrive) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 1 && arrive) mbar_arrive(&bar);
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0, timeout_ns)) atomicOr(&g_tc_error, 1);
}
}  // namespace

cudaError_t tc_timeout_probe_launch(uint64_t timeout_ns, int arrive, cudaStream_t st) {
  timeout_probe_kernel<<<1, 32, 0, st>>>(timeout_ns, arrive);
  return cudaGetLastError();
}

int tc_read_and_clear_error(cudaStream_t st) {
  int h = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_tc_error, sizeof(int), 0, cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return -1;
  if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) !=
        cudaSuccess)
      return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  }
  return h;
}

}  // namespace sanatan
