// Pieces shared by the power-attention forward (chunk_pow_tc.cu) and its
// backward (chunk_pow_bwd_tc.cu): the per-chunk workspace layout written by
// the preparation kernel, and the integer power.
#pragma once
#include <cstdint>

#include "tc_common.cuh"

namespace sanatan {
namespace powc {

using namespace tcc;

// Chunk layouts in the workspace and in shared memory (canonical no-swizzle
// core matrices of 8 rows x 16 bytes):
//   Phi: token group tg (8 tokens) at tg * kXQ, feature group fg (8 features)
//        at fg * 128, token row r at r * 16   (80 KB per chunk)
//   V:   [V | 1 | 0] (80 columns: the ones column makes the tensor core sum
//        the weights, i.e. the denominator, next to the outputs): token group
//        tg at tg * 1280, column group ng (8 columns) at ng * 128, token row r
//        at r * 16                             (20 KB per chunk)
constexpr uint32_t kPhiBytes = 16 * kXQ;   // 81920
constexpr uint32_t kVGroup = 10 * 128;     // bytes per 8-token group of [V | 1 | 0]
constexpr uint32_t kVBytes = 16 * kVGroup; // 20480
constexpr int kNV = 80;                    // N of the value product
constexpr uint32_t kChunkBytes = 2 * kPhiBytes + kVBytes;

// Byte offset of (token t, feature group fg) in a Phi chunk.
__host__ __device__ constexpr uint32_t phi_offset(int t, int fg) {
  return (t >> 3) * kXQ + fg * 128 + (t & 7) * 16;
}

__device__ __forceinline__ const unsigned char* chunk_base(const unsigned char* ws, int64_t bh,
                                                           int nchunks, int c) {
  return ws + (bh * nchunks + c) * static_cast<int64_t>(kChunkBytes);
}

template <int P>
__device__ __forceinline__ float pow_int(float x) {
  if constexpr (P <= 0) {
    return 1.0f;
  } else if constexpr (P == 1) {
    return x;
  } else {
    const float h = pow_int<P / 2>(x);
    return (P & 1) ? h * h * x : h * h;
  }
}

}  // namespace powc
}  // namespace sanatan
