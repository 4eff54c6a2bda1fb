// Pieces shared by the tensor-core kernels of the forward (chunk_tc.cu) and
// the backward (chunk_bwd_tc.cu): chunk and feature geometry, the canonical
// shared-memory operand layouts, the bf16 feature map of eight dimensions,
// and the workspace layout of per-segment state sums.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "sanatan_math.cuh"
#include "tc_ptx.cuh"

namespace sanatan {
namespace tcc {

using namespace tc;

constexpr int kD = 64;
constexpr int kC = 128;              // tokens per chunk (= MMA M)
constexpr int kNF = 320;             // non-constant features
constexpr int kSCRows = kNF + 1;     // + the [sum v | count] row
constexpr int kSCCols = 80;          // compact state row stride (floats)
// Per-segment state sums in the workspace: 68 columns (S, z, 3 pad) of 321
// rows, stored per 128-row tile column-major with the row index fastest, so
// that the threads of a warp (one row each) read and write consecutive words.
constexpr int kSCUsedCols = 68;
__host__ __device__ constexpr int sc_tile_rows(int mt) { return mt < 2 ? 128 : kSCRows - 256; }
// First chunk of segment `seg` when nchunks chunks are split into nseg
// segments (nseg <= nchunks; seg = nseg gives nchunks).  Rounded up, so the
// longer shares go to the first segments: segment 0 needs no earlier sums and
// starts at once, while every later segment waits for the whole state-only
// pass, so an extra chunk costs least there (16 chunks in 3 segments: 6, 5, 5).
// Every kernel that reads or writes per-segment sums uses this split.
__host__ __device__ constexpr int seg_begin(int seg, int nchunks, int nseg) {
  return static_cast<int>((static_cast<long long>(seg) * nchunks + nseg - 1) / nseg);
}
static_assert(seg_begin(1, 16, 3) == 6 && seg_begin(2, 16, 3) == 11 && seg_begin(3, 16, 3) == 16,
              "segment split");
__host__ __device__ constexpr int sc_index(int f, int col) {
  return kSCUsedCols * (f & ~127) + col * sc_tile_rows(f >> 7) + (f & 127);
}
static_assert(kSCUsedCols * kSCRows <= kSCRows * kSCCols, "slot layout must fit the slot");
constexpr int kXQ = 40 * 128;        // bytes per 8-token group of PhiQ
constexpr int kXK = 41 * 128;        // PhiK: + the ones feature group (fg 40)
constexpr int kNG = 9;               // stored 8-column groups of [V | 1 | 0]
constexpr int kLBO_SV = kNG * 128;   // K-direction core stride of S'bf16 and V
constexpr int kN = 80;               // N of the value-side products


// Non-constant feature index f <-> (dimension a, channel c in 1..5).  Features
// are ordered by groups of 8 dimensions: f = 40 * (a / 8) + 8 * (c - 1) + a % 8,
// so any 80 consecutive features hold every channel of 16 dimensions.
__host__ __device__ constexpr int feat_group(int ag, int c) { return 5 * ag + (c - 1); }
__device__ __forceinline__ void feat_dim_chan(int f, int& a, int& c) {
  const int fg = f >> 3;
  a = 8 * (fg / 5) + (f & 7);
  c = fg % 5 + 1;
}

__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


// Eight dimensions of one token: the five non-constant channels, packed as
// bf16 pairs (out[c][j/2] holds dims j, j+1 of channel c).
__device__ __forceinline__ void features8(uint4 raw, const float4* __restrict__ dimc,
                                          const float (&cb)[8], const float (&sb)[8],
                                          uint32_t (&out)[5][4]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    float ch[5][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = 2 * p + h;
      const float u = __uint_as_float((h == 0 ? (w[p] << 16) : (w[p] & 0xffff0000u)));
      const float th = kPi * __fdividef(u, 1.0f + fabsf(u));
      float s, c;
      __sincosf(th, &s, &c);
      const float4 kc = dimc[j];
      const float r = tanh_fast(fmaf(kc.x, c, -kc.y * s));
      const float cr = fmaf(c, cb[j], -s * sb[j]);
      const float sr = fmaf(s, cb[j], c * sb[j]);
      ch[0][h] = cr;
      ch[1][h] = sr;
      ch[2][h] = r;
      ch[3][h] = r * cr;
      ch[4][h] = r * sr;
    }
#pragma unroll
    for (int c = 0; c < 5; ++c) out[c][p] = pack_bf16x2(ch[c][0], ch[c][1]);
  }
}

// The non-constant channels of eight dimensions of one token for the
// feature map with CH channels per dimension, packed as bf16 pairs
// (out[c][j/2] holds dims j, j+1 of channel c), then the rotation of
// (cb, sb) to the thread's next token:
//   CH = 6: cos, sin, r, r cos, r sin  (the six-channel map, eq. (6))
//   CH = 4: r, r cos, r sin            (the four-channel map)
//   CH = 3: cos, sin                   (the three-channel map, no root)
// with cos, sin of the rotated angle and r from the un-rotated one.
template <int CH>
__device__ __forceinline__ void features8_map(uint4 raw, const float4* __restrict__ dimc,
                                              float (&cb)[8], float (&sb)[8],
                                              uint32_t (&out)[CH - 1][4]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    float ch[CH - 1][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = 2 * p + h;
      const float u = __uint_as_float((h == 0 ? (w[p] << 16) : (w[p] & 0xffff0000u)));
      const float th = __fdividef(u, fmaf(fabsf(u), 0.318309886183790672f, 0.318309886183790672f));
      float s, c;
      __sincosf(th, &s, &c);
      const float4 kc = dimc[j];
      const float cr = fmaf(c, cb[j], -s * sb[j]);
      const float sr = fmaf(s, cb[j], c * sb[j]);
      if constexpr (CH == 3) {
        ch[0][h] = cr;
        ch[1][h] = sr;
      } else {
        const float r = tanh_fast(fmaf(kc.x, c, -kc.y * s));
        if constexpr (CH == 6) {
          ch[0][h] = cr;
          ch[1][h] = sr;
          ch[2][h] = r;
          ch[3][h] = r * cr;
          ch[4][h] = r * sr;
        } else {
          ch[0][h] = r;
          ch[1][h] = r * cr;
          ch[2][h] = r * sr;
        }
      }
      const float nc = fmaf(cb[j], kc.z, -sb[j] * kc.w);
      sb[j] = fmaf(sb[j], kc.z, cb[j] * kc.w);
      cb[j] = nc;
    }
#pragma unroll
    for (int c = 0; c < CH - 1; ++c) out[c][p] = pack_bf16x2(ch[c][0], ch[c][1]);
  }
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

}  // namespace tcc
}  // namespace sanatan
