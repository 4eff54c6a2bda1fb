// One decode token through a stack of attention layers (the reading notes'
// §2.7: the whole-model recurrence updates the layers' states in order, each
// layer with its own weights, at the same positions; §3.1: 12 layers of 12
// heads x 64).  The attention path only: per layer
//   q, k, v = x Wq, x Wk, x Wv;  o = the p = 1 decode step of every head;
//   x <- x + o Wo,
// float32 throughout.  Per layer: the projection product into q | k | v, the
// decode step of decode.cu for the layer's B x heads slots, and the output
// product accumulated onto x (the residual) -- 3 launches and a memset.
#include "sanatan_internal.h"

namespace sanatan {
namespace {

constexpr int kMaxB = 8;       // sequences per call
constexpr int kRowsPerCta = 32;

// y[b, col] += sum_k x[b, k] W[k, col] for a 128-column block and 32 rows of
// W per CTA (one warp, four columns per lane, float4 loads), accumulated with
// atomics.  Column col of W goes to y + (col / ysplit) * B * ysplit +
// b * ysplit + col % ysplit (q | k | v split into three [B, ysplit] blocks, or
// ysplit = N for a plain [B, N] output).
__global__ void __launch_bounds__(32) gemv_acc_kernel(const float* __restrict__ x, int B, int K,
                                                      const float* __restrict__ W, int N,
                                                      int ysplit, float* __restrict__ y) {
  __shared__ float xs[kMaxB][kRowsPerCta];
  const int lane = threadIdx.x;
  const int c0 = blockIdx.x * 128 + 4 * lane;
  const int k0 = blockIdx.y * kRowsPerCta;
  const int nk = min(kRowsPerCta, K - k0);
#pragma unroll
  for (int b = 0; b < kMaxB; ++b) xs[b][lane] = (b < B && lane < nk) ? x[b * K + k0 + lane] : 0.f;
  __syncwarp();
  float acc[kMaxB][4];
#pragma unroll
  for (int b = 0; b < kMaxB; ++b)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[b][j] = 0.f;
  // Every row's load is issued before the first product, so that a CTA keeps
  // its whole 16 KB block of W in flight.
  float4 w[kRowsPerCta];
#pragma unroll
  for (int r = 0; r < kRowsPerCta; ++r)
    w[r] = r < nk ? __ldg(reinterpret_cast<const float4*>(W + static_cast<int64_t>(k0 + r) * N + c0))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < kRowsPerCta; ++r) {
#pragma unroll
    for (int b = 0; b < kMaxB; ++b) {
      const float xv = xs[b][r];
      acc[b][0] = fmaf(xv, w[r].x, acc[b][0]);
      acc[b][1] = fmaf(xv, w[r].y, acc[b][1]);
      acc[b][2] = fmaf(xv, w[r].z, acc[b][2]);
      acc[b][3] = fmaf(xv, w[r].w, acc[b][3]);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int col = c0 + j;
    const int64_t base = static_cast<int64_t>(col / ysplit) * B * ysplit + col % ysplit;
#pragma unroll
    for (int b = 0; b < kMaxB; ++b)
      if (b < B) atomicAdd(y + base + static_cast<int64_t>(b) * ysplit, acc[b][j]);
  }
}

cudaError_t gemv_acc(const float* x, int B, int K, const float* W, int N, int ysplit, float* y,
                     cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(N / 128),
                  static_cast<unsigned>((K + kRowsPerCta - 1) / kRowsPerCta));
  gemv_acc_kernel<<<grid, 32, 0, st>>>(x, B, K, W, N, ysplit, y);
  return cudaGetLastError();
}

}  // namespace

size_t stack_workspace_bytes(int B, int heads, int d) {
  return static_cast<size_t>(4) * B * heads * d * sizeof(float);   // q | k | v and o
}

int stack_max_batch() { return kMaxB; }

cudaError_t stack_decode_launch(const StackArgs& a, cudaStream_t st) {
  const int Dm = a.heads * 64;
  const int64_t per_layer_state = static_cast<int64_t>(a.B) * a.heads * 384 * 64;
  float* qkv = static_cast<float*>(a.workspace);
  float* o = qkv + static_cast<int64_t>(3) * a.B * Dm;
  cudaError_t e;
  for (int l = 0; l < a.L; ++l) {
    if ((e = cudaMemsetAsync(qkv, 0, sizeof(float) * 3 * a.B * Dm, st)) != cudaSuccess) return e;
    if ((e = gemv_acc(a.x, a.B, Dm, a.Wqkv + static_cast<int64_t>(l) * Dm * 3 * Dm, 3 * Dm, Dm,
                      qkv, st)) != cudaSuccess)
      return e;
    const float* q = qkv;
    const float* k = qkv + static_cast<int64_t>(a.B) * Dm;
    const float* v = qkv + static_cast<int64_t>(2) * a.B * Dm;
    if ((e = decode_step_launch(a.S + l * per_layer_state, a.z + l * per_layer_state / 64, q, k, v,
                                a.gamma + l * a.heads, a.omega + static_cast<int64_t>(l) * a.heads * 64,
                                a.phi + static_cast<int64_t>(l) * a.heads * 64, a.pos,
                                a.B * a.heads, a.heads, a.eps, o, st)) != cudaSuccess)
      return e;
    if ((e = gemv_acc(o, a.B, Dm, a.Wo + static_cast<int64_t>(l) * Dm * Dm, Dm, Dm, a.x, st)) !=
        cudaSuccess)
      return e;
  }
  return cudaSuccess;
}

}  // namespace sanatan
