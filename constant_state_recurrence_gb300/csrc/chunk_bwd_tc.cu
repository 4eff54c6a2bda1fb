// Backward of the chunked p=1 attention on the tensor cores (bf16 operands,
// f32 accumulation).
//
// The pages give no gradient; this is the chain rule through eqs. (2)-(6) and
// (9) of "SANATAN: Root-Parity Gated Angular Attention with an Exact
// Constant-State Recurrent Form" (reading notes §2.2-§2.7).  With
// dN_t = dO_t / (D_t + eps) and dD_t = -(dO_t . o_t) / (D_t + eps), the three
// gradients are causal linear attentions of their own:
//   dPhi(q_t) = sum_{j<=t} ([dN_t|dD_t] . [v_j|1]) Phi(k_j) + [S|z]_{<chunk} [dN_t|dD_t]
//             = [S|z]_t [dN_t|dD_t]        (the forward state, read with [dN|dD])
//   dPhi(k_j) = sum_{t>=j} ([v_j|1] . [dN_t|dD_t]) Phi(q_t)   (reverse time)
//   dv_j      = sum_{t>=j} (Phi(k_j) . Phi(q_t)) dN_t        (reverse time)
// The first two have 80-wide queries and keys and the 320 non-constant
// features as values ("feature-space attention", this file); dv is the
// forward kernel itself run in reverse with q and k swapped, values dN and
// no normalisation.  Reverse time maps processing position u to row T-1-u and
// keeps each row's own position, so every feature equals the forward's.
//
// Feature-space attention, per chunk of 128 tokens (M = 128 query rows):
//   dS      = Q' K'^T          (Q' = [vq | eq], K' = [vk | ek], K = 80), masked j <= u
//   out_qq  = dS Phi(uk)_qq + Q' [S|z]_qq^T   for the four 80-feature quarters
//   [S|z]  += Phi(uk)^T K'
// out_qq holds dPhi of 16 dimensions; the featuriser warps drain it from TMEM
// and apply the chain rule through the feature map of `ue` (q for dq, k for
// dk), accumulating dgamma, domega, dphi.
#include <cuda_fp16.h>

#include "sanatan_internal.h"
#include "sanatan_math.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace sanatan {

__device__ int g_bwd_tc_error;  // set when a bounded wait gives up

namespace {

using namespace tc;
using namespace tcc;

constexpr int kXA = 10 * 128;  // Q' = [vq | eq | 0]: bytes per 8-token group (K-major, K = 80)

constexpr uint32_t kTD = 0;     // TMEM: dS (f32, 128 cols) / dS~ (bf16, cols 0..63)
constexpr uint32_t kTQ = 128;   // TMEM: one 80-feature quarter of dPhi
constexpr uint32_t kTS = 208;   // TMEM: state tiles at 208, 288, 368
constexpr uint32_t kTmemCols = 512;

constexpr int kOffF = 0;                        // Phi(uk): 16 token groups x kXK
constexpr int kOffS = kOffF + 16 * kXK;         // state snapshot bf16: 40 x kLBO_SV
constexpr int kOffQ = kOffS + 40 * kLBO_SV;     // Q'
constexpr int kOffV = kOffQ + 16 * kXA;         // K' = [vk | ek | 0] (+ over-read pad)
// Rotation factors cos(t phi_a), sin(t phi_a) of the chunk's tokens as f16
// pairs, written while staging and read by the chain rule (rows padded to 272 B
// so that row-per-lane reads spread over the banks).
constexpr int kRotPitch = 272;
constexpr int kOffR = kOffV + 16 * kLBO_SV + 128;
constexpr int kOffMisc = kOffR + kC * kRotPitch;

enum Bar {
  kFeatFull = 0, kSFull, kSTilde, kOutFull, kOutFree, kStateDone, kSnapReady, kDrain, kNumBars
};

struct Misc {
  float4 dimc[64];   // featuriser constants (as the forward kernel)
  float4 pc[64];     // chain rule: cos omega, sin omega, phi, 0
  float gacc[2 * 64 + 4];  // domega (64), dphi (64), dgamma
  uint64_t bar[kNumBars];
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int kSmemBytes = kOffMisc + static_cast<int>(sizeof(Misc));
static_assert(kSmemBytes <= 232448, "shared memory layout exceeds 227 KB");

// 768 threads: warps 0-15 stage the chunk and apply the chain rule (the
// launch allocation of 80 registers), warps 16-19 drain TMEM (128 registers
// after setmaxnreg), one thread of warp 20 issues the MMAs (its warpgroup
// keeps 32).
constexpr int kThreads = 768;
constexpr uint32_t kRegLaunch = 80;
constexpr uint32_t kRegEpi = 128;
constexpr uint32_t kRegMma = 32;
static_assert(512 * kRegLaunch + 128 * kRegEpi + 128 * kRegMma <= kThreads * kRegLaunch,
              "setmaxnreg split must fit the launch allocation");
constexpr int kFeatWarps = 16;
constexpr int kEpiWarp0 = 16;
constexpr int kMmaWarp = 20;
constexpr uint64_t kWaitNs = 2000000000ull;

struct FsaParams {
  const __nv_bfloat16* uk;  // raw u whose features are the values (k for dq, q for dk)
  const __nv_bfloat16* ue;  // raw u the gradient is for (q for dq, k for dk)
  const __nv_bfloat16* vq;  // query rows [T x 64] (dN for dq, v for dk)
  const float* eq;          // query extra column (dD for dq, null = 1 for dk)
  const __nv_bfloat16* vk;  // key rows (v for dq, dN for dk)
  const float* ek;          // key extra column (null = 1 for dq, dD for dk)
  const float* gamma;
  const float* omega;
  const float* phi;
  int H, T;
  int64_t pos0;
  int reverse;
  int nseg, seg_grid, nchunks;
  const float* deltas;      // per-segment state sums (sc_index layout) or null
  const float* S0;          // caller's initial state (dq only) or null
  const float* z0;
  __nv_bfloat16* du;        // output [B, H, T, 64]
  float* dgamma;            // [H], accumulated
  float* domega;            // [H, 64], accumulated
  float* dphi;              // [H, 64], accumulated (may be null)
};

__device__ __forceinline__ bool wait_bar(Misc& m, int b, uint32_t parity) {
  if (*reinterpret_cast<volatile int*>(&m.abort_flag)) return false;
  if (mbar_wait_bounded(&m.bar[b], parity, kWaitNs)) return true;
  m.abort_flag = 1;
  atomicOr(&g_bwd_tc_error, 1);
  return false;
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void feat_sync() { asm volatile("bar.sync 2, 512;" ::: "memory"); }

// L2 prefetch of one chunk's rows of uk, ue, the query and key rows and the
// extra columns (sizes rounded down to whole 16-byte pieces).
__device__ __forceinline__ void prefetch_chunk_rows(const FsaParams& prm, int64_t seq_row0, int chunk) {
  const int tok0 = chunk * kC;
  const int n = min(kC, prm.T - tok0);
  if (n <= 0) return;
  const int64_t row = seq_row0 + (prm.reverse ? prm.T - tok0 - n : tok0);
  const uint32_t bytes = static_cast<uint32_t>(n) * kD * 2;
  prefetch_l2_bulk(prm.uk + row * kD, bytes);
  prefetch_l2_bulk(prm.ue + row * kD, bytes);
  prefetch_l2_bulk(prm.vq + row * kD, bytes);
  prefetch_l2_bulk(prm.vk + row * kD, bytes);
  const uint32_t xb = (static_cast<uint32_t>(n) * 4) & ~15u;
  const float* x = prm.eq != nullptr ? prm.eq : prm.ek;
  if (x != nullptr && xb > 0 && ((reinterpret_cast<uintptr_t>(x + row) & 15u) == 0))
    prefetch_l2_bulk(x + row, xb);
}

__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ int frow(const FsaParams& p, int u) {
  return p.reverse ? p.T - 1 - u : u;
}

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

// Reduce 8 per-lane values over the 32 lanes of a warp: afterwards the four
// lanes 4i..4i+3 hold the total of value index slot8(i), with slot taken from
// lane bits 4..2.
__device__ __forceinline__ float warp_reduce8(float (&v)[8], int lane) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool up = lane & 16;
    const float send = up ? v[i] : v[i + 4];
    const float keep = up ? v[i + 4] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool up = lane & 8;
    const float send = up ? v[i] : v[i + 2];
    const float keep = up ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  {
    const bool up = lane & 4;
    const float send = up ? v[0] : v[1];
    const float keep = up ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  float t = v[0] + __shfl_xor_sync(0xffffffffu, v[0], 2);
  return t + __shfl_xor_sync(0xffffffffu, t, 1);
}
__device__ __forceinline__ int reduce8_slot(int lane) {
  return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
}
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) fsa_kernel(FsaParams prm) {
  extern __shared__ __align__(1024) unsigned char smem[];
  Misc& m = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const uint32_t sF = smem_u32(smem + kOffF);
  const uint32_t sS = smem_u32(smem + kOffS);
  const uint32_t sQ = smem_u32(smem + kOffQ);
  const uint32_t sV = smem_u32(smem + kOffV);
  const uint32_t sR = smem_u32(smem + kOffR);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int bh = blockIdx.x / prm.seg_grid;
  const int seg = blockIdx.x % prm.seg_grid;
  const int h = bh % prm.H;
  const int c_begin = seg_begin(seg, prm.nchunks, prm.nseg);
  const int c_end = seg_begin(seg + 1, prm.nchunks, prm.nseg);
  const int nloc = c_end - c_begin;
  const int64_t seq_row0 = static_cast<int64_t>(bh) * prm.T;

  if (warp == kMmaWarp) {
    tmem_alloc(&m.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b) {
      const uint32_t cnt = (b == kFeatFull || b == kOutFree) ? kFeatWarps
                           : (b == kSTilde || b == kSnapReady) ? 4u : 1u;
      mbar_init(&m.bar[b], cnt);
    }
    m.abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < kD) {
    const float g = prm.gamma[h] * 1.41421356237309515f;
    const float om = prm.omega[h * kD + tid];
    const float ph = prm.phi[h * kD + tid];
    float sw, cw;
    sincosf(om + 0.785398163397448310f, &sw, &cw);
    float s8, c8;
    sincosf(phase_mod_2pi(8, ph), &s8, &c8);
    m.dimc[tid] = make_float4(g * cw, g * sw, c8, prm.reverse ? -s8 : s8);
    float so, co;
    sincosf(om, &so, &co);
    m.pc[tid] = make_float4(co, so, ph, 0.f);
  }
  for (int i = tid; i < 2 * 64 + 4; i += kThreads) m.gacc[i] = 0.f;
  // Constant parts of Q' (column groups 8, 9) and K' (column group 8) when the
  // extra column is one; per-token values are written per chunk otherwise.
  if (tid < 128) {
    const int tg = tid >> 3, r = tid & 7;
    st_shared_v4(sQ + tg * kXA + 8 * 128 + r * 16, prm.eq ? 0u : 0x3F80u, 0u, 0u, 0u);
    st_shared_v4(sQ + tg * kXA + 9 * 128 + r * 16, 0u, 0u, 0u, 0u);
    st_shared_v4(sV + tg * kLBO_SV + 8 * 128 + r * 16, prm.ek ? 0u : 0x3F80u, 0u, 0u, 0u);
  }
  if (tid < 8) st_shared_v4(sV + 16 * kLBO_SV + 16 * tid, 0u, 0u, 0u, 0u);  // over-read pad
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;
  float acc_gamma = 0.f;

  if (warp < kFeatWarps) {
    // ------------------------------------------------- featuriser + chain rule
    // Staging role: lane (r, dimension group ag) of warp w owns tokens
    // tq + 8 i (i = 0, 1) of the chunk.
    const int fw = warp & 7;
    const int r = lane & 7;
    const int ag = (lane >> 3) + 4 * (fw & 1);
    const int tq = 32 * (fw >> 1) + r + 16 * (warp >> 3);
    const float4* dimc = &m.dimc[8 * ag];
    // chain-rule role: TMEM lane quarter lq, and four dimensions (4 sub) of
    // each quarter's sixteen
    const int lq = warp & 3;
    const int sub = warp >> 2;
    const int crow = 32 * lq + lane;   // token row of the chunk
    const float gam = prm.gamma[h];

    // Raw uk, query and key rows of one chunk for this thread's two tokens.
    // They are loaded right after the chunk's staging hand-off (an arrive with
    // release semantics would wait for loads still in flight) and consumed when
    // the next chunk is staged.
    uint4 ru[2], rq[2], rk[2];
    float xq[2], xk[2];  // extra columns (read by the ag == 0 lanes)
    auto load_stage = [&](int chunk) {
      const int tok0 = chunk * kC;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t = tq + 8 * i;
        const bool valid = chunk < c_end && tok0 + t < prm.T;
        const int64_t row = seq_row0 + frow(prm, valid ? tok0 + t : 0);
        const int64_t off = row * kD + 8 * ag;
        ru[i] = valid ? ldg_nc_v4(prm.uk + off) : make_uint4(0u, 0u, 0u, 0u);
        rq[i] = valid ? ldg_nc_v4(prm.vq + off) : make_uint4(0u, 0u, 0u, 0u);
        rk[i] = valid ? ldg_nc_v4(prm.vk + off) : make_uint4(0u, 0u, 0u, 0u);
        xq[i] = (valid && ag == 0 && prm.eq != nullptr) ? __ldg(prm.eq + row) : 0.f;
        xk[i] = (valid && ag == 0 && prm.ek != nullptr) ? __ldg(prm.ek + row) : 0.f;
      }
    };
    if (tid == 0) {
      if (nloc > 0) prefetch_chunk_rows(prm, seq_row0, c_begin);
      if (nloc > 1) prefetch_chunk_rows(prm, seq_row0, c_begin + 1);
    }
    load_stage(c_begin);
    for (int ci = 0; ci < nloc; ++ci) {
      const int chunk = c_begin + ci;
      const int tok0 = chunk * kC;
      if (tid == 0 && ci + 2 < nloc) prefetch_chunk_rows(prm, seq_row0, chunk + 2);
      // --- stage Phi(uk), Q', K' of the chunk
      float cb[8], sb[8];
      {
        const int64_t tabs = prm.pos0 + frow(prm, tok0 + tq);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          __sincosf(phase_mod_2pi(tabs, m.pc[8 * ag + j].z), &sb[j], &cb[j]);
      }
      if (ci > 0) wait_bar(m, kStateDone, (ci - 1) & 1);
      feat_sync();  // every chain-rule read of the previous chunk's rotation table is done
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t = tq + 8 * i;
        const bool valid = tok0 + t < prm.T;
        uint32_t kf[5][4];
        if (valid) {
          features8(ru[i], dimc, cb, sb, kf);
        } else {
#pragma unroll
          for (int c = 0; c < 5; ++c)
#pragma unroll
            for (int p = 0; p < 4; ++p) kf[c][p] = 0u;
        }
        const uint32_t base = sF + (t >> 3) * kXK + (t & 7) * 16;
#pragma unroll
        for (int c = 0; c < 5; ++c)
          st_shared_v4(base + feat_group(ag, c + 1) * 128, kf[c][0], kf[c][1], kf[c][2], kf[c][3]);
        st_shared_v4(sQ + (t >> 3) * kXA + ag * 128 + (t & 7) * 16, rq[i].x, rq[i].y, rq[i].z,
                     rq[i].w);
        st_shared_v4(sV + (t >> 3) * kLBO_SV + ag * 128 + (t & 7) * 16, rk[i].x, rk[i].y,
                     rk[i].z, rk[i].w);
        // rotation factors of token t, dimensions 8 ag .. 8 ag + 7
        const uint32_t rb = sR + t * kRotPitch + ag * 32;
        st_shared_v4(rb, pack_half2(cb[0], sb[0]), pack_half2(cb[1], sb[1]),
                     pack_half2(cb[2], sb[2]), pack_half2(cb[3], sb[3]));
        st_shared_v4(rb + 16, pack_half2(cb[4], sb[4]), pack_half2(cb[5], sb[5]),
                     pack_half2(cb[6], sb[6]), pack_half2(cb[7], sb[7]));
        if (ag == 0) {
          if (prm.eq != nullptr)
            st_shared_v4(sQ + (t >> 3) * kXA + 8 * 128 + (t & 7) * 16,
                         __bfloat16_as_ushort(__float2bfloat16_rn(xq[i])), 0u, 0u, 0u);
          if (prm.ek != nullptr)
            st_shared_v4(sV + (t >> 3) * kLBO_SV + 8 * 128 + (t & 7) * 16,
                         __bfloat16_as_ushort(__float2bfloat16_rn(xk[i])), 0u, 0u, 0u);
        }
        if (i == 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 kc = dimc[j];
            const float nc = fmaf(cb[j], kc.z, -sb[j] * kc.w);
            sb[j] = fmaf(sb[j], kc.z, cb[j] * kc.w);
            cb[j] = nc;
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&m.bar[kFeatFull]);
      load_stage(chunk + 1);
      feat_sync();  // the rotation table of this chunk is complete

      // --- chain rule for the four quarters of dPhi of this chunk
      const int u = tok0 + crow;
      const bool rvalid = u < prm.T;
      const int64_t grow = seq_row0 + frow(prm, rvalid ? u : 0);
      const int64_t tpos = prm.pos0 + frow(prm, rvalid ? u : 0);
      const float tposf = static_cast<float>(tpos);
      // dimensions a0 .. a0 + 3 of quarter qq: a0(qq) = 16 qq + 8 (sub / 2) + 4 (sub % 2)
      const int a_sub = 8 * (sub >> 1) + 4 * (sub & 1);
      // raw u of this row, one quarter ahead of its use
      uint2 raw_next = rvalid ? ldg_nc_v2(prm.ue + grow * kD + a_sub) : make_uint2(0u, 0u);
#pragma unroll 1
      for (int qq = 0; qq < 4; ++qq) {
        const int a0 = 16 * qq + a_sub;
        const uint2 raw = raw_next;
        if (qq < 3)
          raw_next = rvalid ? ldg_nc_v2(prm.ue + grow * kD + a0 + 16) : make_uint2(0u, 0u);
        wait_bar(m, kOutFull, (4 * ci + qq) & 1);
        tc_fence_after();
        float dphi5[5][4];
        const uint32_t ta = tmem + (static_cast<uint32_t>(32 * lq) << 16) + kTQ + 40 * (sub >> 1) +
                            4 * (sub & 1);
#pragma unroll
        for (int c = 0; c < 5; ++c) tmem_ld4(ta + 8 * c, dphi5[c]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(&m.bar[kOutFree]);  // the quarter is in registers
        // rotation factors of this row for dimensions a0 .. a0 + 3
        uint32_t rot[4];
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(rot[0]), "=r"(rot[1]), "=r"(rot[2]), "=r"(rot[3])
                     : "r"(sR + crow * kRotPitch + a0 * 4));
        const uint32_t w[2] = {raw.x, raw.y};
        float red[8];
        uint32_t outp[2];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float uu = __uint_as_float((j & 1) ? (w[j >> 1] & 0xffff0000u) : (w[j >> 1] << 16));
          const float inv = __fdividef(1.0f, 1.0f + fabsf(uu));
          const float th = kPi * (uu * inv);
          float st, ct;
          __sincosf(th, &st, &ct);
          const float4 pc = m.pc[a0 + j];
          const float cx = ct * pc.x - st * pc.y;   // cos(theta + omega)
          const float sx = st * pc.x + ct * pc.y;   // sin(theta + omega)
          const float gx = cx - sx;
          const float gpx = -sx - cx;
          const float rr = tanh_fast(gam * gx);
          const float2 rcs = __half22float2(*reinterpret_cast<const __half2*>(&rot[j]));
          const float cp = rcs.x, sp = rcs.y;
          const float cr = ct * cp - st * sp;
          const float sr = st * cp + ct * sp;
          const float d1 = dphi5[0][j], d2 = dphi5[1][j], d3 = dphi5[2][j];
          const float d4 = dphi5[3][j], d5 = dphi5[4][j];
          const float dc = fmaf(rr, d4, d1);
          const float ds = fmaf(rr, d5, d2);
          const float dr = d3 + cr * d4 + sr * d5;
          const float dth_rot = ds * cr - dc * sr;
          const float dpre = dr * (1.0f - rr * rr);
          const float dtheta = fmaf(dpre * gam, gpx, dth_rot);
          const float du = rvalid ? dtheta * (kPi * inv * inv) : 0.f;
          if (j & 1)
            outp[j >> 1] |= static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(du))) << 16;
          else
            outp[j >> 1] = __bfloat16_as_ushort(__float2bfloat16_rn(du));
          red[j] = rvalid ? dpre * gam * gpx : 0.f;   // domega
          red[4 + j] = rvalid ? dth_rot * tposf : 0.f; // dphi
          acc_gamma += rvalid ? dpre * gx : 0.f;
        }
        if (rvalid) *reinterpret_cast<uint2*>(prm.du + grow * kD + a0) = make_uint2(outp[0], outp[1]);
        const float tot = warp_reduce8(red, lane);
        if ((lane & 3) == 0) {
          const int slot = reduce8_slot(lane);
          atomicAdd(&m.gacc[(slot < 4 ? 0 : 64) + a0 + (slot & 3)], tot);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc_gamma += __shfl_xor_sync(0xffffffffu, acc_gamma, off);
    if (lane == 0) atomicAdd(&m.gacc[128], acc_gamma);
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------- TMEM epilogue
    setmaxnreg_inc<kRegEpi>();
    const int qd = warp - kEpiWarp0;
    const int row = 32 * qd + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
    // Initial state: caller's (S0, z0) plus the sums of earlier segments.
    for (int mt = 0; mt < 3; ++mt) {
      const int f = mt * 128 + row;
      if (mt == 2 && qd == 3) continue;
      float val[80];
#pragma unroll
      for (int e = 0; e < 80; ++e) val[e] = 0.f;
      if (f < kNF && prm.S0 != nullptr) {
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
      if (f < kSCRows && prm.deltas != nullptr) {
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
      if (f < kNF) {
        const uint32_t base = sS + (f >> 3) * kLBO_SV + (f & 7) * 16;
#pragma unroll
        for (int ng = 0; ng < kNG; ++ng)
          st_shared_v4(base + ng * 128, pack_bf16x2(val[8 * ng], val[8 * ng + 1]),
                       pack_bf16x2(val[8 * ng + 2], val[8 * ng + 3]),
                       pack_bf16x2(val[8 * ng + 4], val[8 * ng + 5]),
                       pack_bf16x2(val[8 * ng + 6], val[8 * ng + 7]));
      }
    }
    tmem_st_wait();
    fence_proxy_async_smem();
    tc_fence_before();
    epi_sync();
    if (lane == 0) mbar_arrive(&m.bar[kSnapReady]);
    for (int ci = 0; ci < nloc; ++ci) {
      // E1: mask dS to j <= u and convert it to bf16 in place (A operand of the quarters).
      wait_bar(m, kSFull, ci & 1);
      tc_fence_after();
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        uint32_t pk[16];
        if (b > qd) {
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = 0u;
        } else {
          float p[32];
          tmem_ld16(tmem + lane_off + kTD + 32 * b, *reinterpret_cast<float(*)[16]>(&p[0]));
          tmem_ld16(tmem + lane_off + kTD + 32 * b + 16, *reinterpret_cast<float(*)[16]>(&p[16]));
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int j0 = 32 * b + 2 * i;
            pk[i] = pack_bf16x2(j0 <= row ? p[2 * i] : 0.f, j0 + 1 <= row ? p[2 * i + 1] : 0.f);
          }
        }
        tmem_st16(tmem + lane_off + kTD + 16 * b, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&m.bar[kSTilde]);
      // E2: bf16 snapshot of the state after this chunk, for the next chunk.
      wait_bar(m, kStateDone, ci & 1);
      tc_fence_after();
      if (ci + 1 < nloc) {
        for (int mt = 0; mt < 3; ++mt) {
          if (mt == 2 && qd >= 2) continue;  // rows 320.. are not needed here
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
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        epi_sync();
        if (lane == 0) mbar_arrive(&m.bar[kSnapReady]);
      }
    }
  } else {
    setmaxnreg_dec<kRegMma>();
  }
  if (warp == kMmaWarp && lane == 0) {
    // ------------------------------------------------- MMA issuer
    constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idOF = idesc_bf16_f32(128, kN, false, true);   // dS~ Phi(uk): B MN-major
    constexpr uint32_t idOS = idesc_bf16_f32(128, kN, false, false);  // Q' S^T: B K-major
    constexpr uint32_t idST = idesc_bf16_f32(128, kN, true, true);
    const uint64_t dQp = smem_desc(sQ, 128, kXA);          // Q', K-major A (K = 80)
    const uint64_t dKp = smem_desc(sV, 128, kLBO_SV);      // K' as K-major B (N = keys)
    const uint64_t dFb = smem_desc(sF, kXK, 128);          // Phi(uk) as MN-major B (N = features)
    const uint64_t dSb = smem_desc(sS, 128, kLBO_SV);      // snapshot as K-major B (N = features)
    const uint64_t dFa = smem_desc(sF, kXK, 128);          // Phi(uk)^T, MN-major A (state)
    const uint64_t dVb = smem_desc(sV, kLBO_SV, 128);      // K' as MN-major B (state)
    for (int ci = 0; ci < nloc; ++ci) {
      uint64_t q0 = dQp, k0 = dKp, f0 = dFb, s0 = dSb, fa = dFa, vb = dVb;
      asm volatile("" : "+l"(q0), "+l"(k0), "+l"(f0), "+l"(s0), "+l"(fa), "+l"(vb));
      wait_bar(m, kFeatFull, ci & 1);
      tc_fence_after();
#pragma unroll
      for (int s = 0; s < 5; ++s) mma_ss(tmem + kTD, q0 + 16 * s, k0 + 16 * s, idS, s > 0);
      mma_commit(&m.bar[kSFull]);
      wait_bar(m, kSTilde, ci & 1);
      wait_bar(m, kSnapReady, ci & 1);
      tc_fence_after();
#pragma unroll 1
      for (int qq = 0; qq < 4; ++qq) {
        const int ph = 4 * ci + qq;
        if (ph > 0) wait_bar(m, kOutFree, (ph - 1) & 1);
        tc_fence_after();
        uint64_t fq = f0 + (10 * 128 / 16) * qq, sq = s0 + (10 * kLBO_SV / 16) * qq;
        asm volatile("" : "+l"(fq), "+l"(sq), "+l"(q0));
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ts(tmem + kTQ, tmem + kTD + 8 * s, fq + (2 * kXK / 16) * s, idOF, s > 0);
#pragma unroll
        for (int s = 0; s < 5; ++s) mma_ss(tmem + kTQ, q0 + 16 * s, sq + 16 * s, idOS, true);
        mma_commit(&m.bar[kOutFull]);
      }
      asm volatile("" : "+l"(fa), "+l"(vb));
#pragma unroll
      for (int s = 0; s < 8; ++s)
#pragma unroll
        for (int mt = 0; mt < 3; ++mt)
          mma_ss(tmem + kTS + mt * kN, fa + (2048 / 16) * mt + (2 * kXK / 16) * s,
                 vb + (2 * kLBO_SV / 16) * s, idST, true);
      mma_commit(&m.bar[kStateDone]);
    }
    // Wait (bounded) for the drain even after an abandoned wait.
    mma_commit(&m.bar[kDrain]);
    mbar_wait_bounded(&m.bar[kDrain], 0, kWaitNs);
  }

  tc_fence_before();
  __syncthreads();
  if (tid < 64) {
    atomicAdd(&prm.domega[h * kD + tid], m.gacc[tid]);
    if (prm.dphi) atomicAdd(&prm.dphi[h * kD + tid], m.gacc[64 + tid]);
  }
  if (tid == 64) atomicAdd(&prm.dgamma[h], m.gacc[128]);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// dN = dO / (D + eps) (bf16) and dD = -(dO . o) / (D + eps) (f32).  Eight
// lanes per row, eight elements per lane (16- and 32-byte accesses).
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&g)[8]) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    g[2 * i] = __uint_as_float(u[i] << 16);
    g[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load8(const float* p, float (&g)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
  g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
}

template <typename Tg>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const Tg* __restrict__ dO,
                                                       const float* __restrict__ o,
                                                       const float* __restrict__ Dn, float eps,
                                                       int64_t rows, __nv_bfloat16* __restrict__ dN,
                                                       float* __restrict__ dD) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 32 + (threadIdx.x >> 3);
  const int part = threadIdx.x & 7;  // elements 8 part .. 8 part + 7 of the row
  const bool ok = row < rows;
  const int64_t r = ok ? row : 0;
  float g[8], ov[8];
  load8(dO + r * 64 + 8 * part, g);
  load8(o + r * 64 + 8 * part, ov);
  const float inv = 1.0f / (Dn[r] + eps);
  float dot = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) dot = fmaf(g[i], ov[i], dot);
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  if (!ok) return;
  *reinterpret_cast<uint4*>(dN + r * 64 + 8 * part) =
      make_uint4(pack_bf16x2(g[0] * inv, g[1] * inv), pack_bf16x2(g[2] * inv, g[3] * inv),
                 pack_bf16x2(g[4] * inv, g[5] * inv), pack_bf16x2(g[6] * inv, g[7] * inv));
  if (part == 0) dD[r] = -dot * inv;
}

}  // namespace

int bwd_tc_read_and_clear_error(cudaStream_t st) {
  int h = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_bwd_tc_error, sizeof(int), 0, cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return -1;
  if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_bwd_tc_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                st) != cudaSuccess)
      return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  }
  return h;
}

size_t chunk_bwd_tc_workspace_bytes(int B, int H, int T) {
  const size_t rows = static_cast<size_t>(B) * H * T;
  const size_t dn = (rows * 64 * 2 + 255) / 256 * 256;
  const size_t dd = (rows * 4 + 255) / 256 * 256;
  const int nseg = tc_segments(B, H, T);
  // One segment reads and writes no per-segment sums.
  const size_t deltas =
      nseg > 1 ? static_cast<size_t>(B) * H * nseg * kSCRows * kSCCols * 4 : 0;
  return dn + dd + 2 * deltas;
}

cudaError_t chunk_bwd_tc_launch(const ChunkBwdArgs& a, cudaStream_t st) {
  const ChunkFwdArgs& f = a.f;
  const int B = f.B, H = f.H, T = f.T;
  cudaError_t e;
  if ((e = cudaMemsetAsync(a.dgamma, 0, sizeof(float) * H, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(a.domega, 0, sizeof(float) * H * kD, st)) != cudaSuccess) return e;
  if (a.dphi && (e = cudaMemsetAsync(a.dphi, 0, sizeof(float) * H * kD, st)) != cudaSuccess)
    return e;
  const int64_t rows = static_cast<int64_t>(B) * H * T;
  if (rows == 0) return cudaSuccess;
  unsigned char* ws = static_cast<unsigned char*>(a.workspace);
  const size_t dn_bytes = (static_cast<size_t>(rows) * 64 * 2 + 255) / 256 * 256;
  const size_t dd_bytes = (static_cast<size_t>(rows) * 4 + 255) / 256 * 256;
  __nv_bfloat16* dN = reinterpret_cast<__nv_bfloat16*>(ws);
  float* dD = reinterpret_cast<float*>(ws + dn_bytes);
  const int nseg = tc_segments(B, H, T);
  const size_t delta_bytes = static_cast<size_t>(B) * H * nseg * kSCRows * kSCCols * 4;
  float* fdeltas = reinterpret_cast<float*>(ws + dn_bytes + dd_bytes);
  float* rdeltas = reinterpret_cast<float*>(ws + dn_bytes + dd_bytes + delta_bytes);

  {
    const unsigned blocks = static_cast<unsigned>((rows + 31) / 32);
    if (a.grad_dtype == SANATAN_F32)
      bwd_prep_kernel<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(a.dO), a.o, a.Dn,
                                                     f.eps, rows, dN, dD);
    else
      bwd_prep_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(
          static_cast<const __nv_bfloat16*>(a.dO), a.o, a.Dn, f.eps, rows, dN, dD);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(f.q);
  const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(f.k);
  const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(f.v);

  // Per-segment sums: forward state sum Phi(k)[v|1] (for dq) and reverse-time
  // sum Phi(q)[dN|dD] (for dk and dv).  The forward-time sums are the ones the
  // forward wrote at the start of its workspace when it used the same split.
  if (nseg > 1) {
    TcJob fs{};
    fs.q = nullptr; fs.k = k; fs.v = v; fs.extra = nullptr;
    fs.gamma = f.gamma; fs.omega = f.omega; fs.phi = f.phi;
    fs.B = B; fs.H = H; fs.T = T; fs.pos0 = f.pos0;
    if (a.fwd_workspace != nullptr && tc_segments_fit(B, H, T, a.fwd_workspace_bytes) == nseg) {
      fdeltas = static_cast<float*>(const_cast<void*>(a.fwd_workspace));
    } else {
      fs.deltas = fdeltas;
      if ((e = tc_state_pass(fs, st)) != cudaSuccess) return e;
    }
    TcJob rs = fs;
    rs.k = q; rs.v = dN; rs.extra = dD; rs.reverse = 1; rs.deltas = rdeltas;
    if ((e = tc_state_pass(rs, st)) != cudaSuccess) return e;
  }
  {
    static bool done[64];
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (!(dev >= 0 && dev < 64 && done[dev])) {
      e = cudaFuncSetAttribute(fsa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) done[dev] = true;
    }
  }
  FsaParams p{};
  p.gamma = f.gamma; p.omega = f.omega; p.phi = f.phi;
  p.H = H; p.T = T; p.pos0 = f.pos0;
  p.nseg = nseg; p.seg_grid = nseg; p.nchunks = (T + kC - 1) / kC;
  p.dgamma = a.dgamma; p.domega = a.domega; p.dphi = a.dphi;
  // dq: forward time, queries [dN|dD], keys [v|1], values Phi(k)
  FsaParams pq = p;
  pq.uk = k; pq.ue = q; pq.vq = dN; pq.eq = dD; pq.vk = v; pq.ek = nullptr;
  pq.reverse = 0; pq.deltas = nseg > 1 ? fdeltas : nullptr; pq.S0 = f.S0; pq.z0 = f.z0;
  pq.du = static_cast<__nv_bfloat16*>(a.dq);
  const ProfileEvents& pe = profile_events();
  if (pe.start != nullptr) cudaEventRecord(pe.start, st);
  fsa_kernel<<<B * H * nseg, kThreads, kSmemBytes, st>>>(pq);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (pe.stop != nullptr) cudaEventRecord(pe.stop, st);
  // dk: reverse time, queries [v|1], keys [dN|dD], values Phi(q)
  FsaParams pk = p;
  pk.uk = q; pk.ue = k; pk.vq = v; pk.eq = nullptr; pk.vk = dN; pk.ek = dD;
  pk.reverse = 1; pk.deltas = nseg > 1 ? rdeltas : nullptr; pk.S0 = nullptr; pk.z0 = nullptr;
  pk.du = static_cast<__nv_bfloat16*>(a.dk);
  fsa_kernel<<<B * H * nseg, kThreads, kSmemBytes, st>>>(pk);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // dv: the forward attention in reverse time with q and k swapped, values dN,
  // no normalisation, bf16 output.
  TcJob dvj{};
  dvj.q = k; dvj.k = q; dvj.v = dN; dvj.extra = dD;
  dvj.gamma = f.gamma; dvj.omega = f.omega; dvj.phi = f.phi;
  dvj.B = B; dvj.H = H; dvj.T = T; dvj.pos0 = f.pos0;
  dvj.o = a.dv; dvj.reverse = 1; dvj.normalize = 0; dvj.out_bf16 = 1;
  dvj.deltas = nseg > 1 ? rdeltas : nullptr; dvj.deltas_ready = 1; dvj.record_events = 0;
  return tc_attention(dvj, st);
}

}  // namespace sanatan
