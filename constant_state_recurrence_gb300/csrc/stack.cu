// One decode token through a stack of attention layers (the reading notes'
// §2.7: the whole-model recurrence updates the layers' states in order, each
// layer with its own weights, at the same positions; §3.1: 12 layers of 12
// heads x 64).  The attention path only: per layer
//   q, k, v = x Wq, x Wk, x Wv;  o = the p = 1 decode step of every head;
//   x <- x + o Wo,
// float32 throughout.
//
// One cooperative launch per token runs every layer: a grid of one CTA per SM
// goes through three phases per layer separated by grid-wide barriers,
//   A  [q | k | v] += x Wqkv  (warp items of 128 columns x 32 rows of W, every
//      row's load issued before the first product, column sums accumulated
//      with float atomics into one of two buffers, the other one zeroed for
//      the next layer),
//   B  the decode step of each slot (CTA items of one slot's 48 feature rows =
//      8 dimensions: state rows updated in place, readout partials of the
//      numerator and denominator accumulated with atomics),
//   C  x += o Wo with o = numerator / (denominator + eps) (warp items of 128
//      columns x 16 rows).
// Data produced inside the kernel (x, q | k | v, the readout sums) is read
// through L2 (ld.global.cg), never from a possibly stale L1 line.  The barriers
// are bounded: a CTA that waits longer than a second records a timeout in the
// library's error word, raises an abort flag that ends every other CTA's wait,
// and returns.
#include "decode_math.cuh"
#include "sanatan_internal.h"
#include "sanatan_math.cuh"

namespace sanatan {

__device__ int g_stack_error;  // set when a grid barrier gives up

namespace {

constexpr int kMaxB = 8;                 // sequences per call
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsA = 32;               // rows of Wqkv per phase-A item
constexpr int kRowsC = 16;               // rows of Wo per phase-C item
constexpr int kParts = 8;                // phase-B items per slot (8 dimensions each)
constexpr int kRowsB = 384 / kParts;     // 48 state rows per item
constexpr uint64_t kBarrierNs = 1000000000ull;

// Workspace: barrier words, then the two [q | k | v] buffers, then the
// readout sums (numerator [N, 64], denominator [N]).
constexpr int kBarWords = 4;             // arrivals, generation, abort, pad

struct FusedParams {
  float* x;
  const float* Wqkv;
  const float* Wo;
  float* S;
  float* z;
  const float* gamma;
  const float* omega;
  const float* phi;
  const int64_t* pos;
  int L, heads;
  float eps;
  unsigned* bar;
  float* qkv;   // [2][3][B][Dm]
  float* num;   // [B * heads][64]
  float* den;   // [B * heads]
};

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void red_add(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Grid-wide barrier of a cooperative launch (every CTA is resident).  `gen`
// counts the barriers this CTA has passed; the generation word starts at 0.
// Returns false after a timeout or another CTA's abort.
__device__ bool grid_sync(unsigned* bar, unsigned& gen) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    const unsigned g = gen;
    if (atomicAdd(&bar[0], 1u) == gridDim.x - 1) {
      atomicExch(&bar[0], 0u);
      __threadfence();
      atomicAdd(&bar[1], 1u);
    } else {
      const uint64_t t0 = now_ns();
      while (*reinterpret_cast<volatile unsigned*>(&bar[1]) == g) {
        if (*reinterpret_cast<volatile unsigned*>(&bar[2]) != 0u) {
          ok = 0;
          break;
        }
        if (now_ns() - t0 > kBarrierNs) {
          atomicExch(&bar[2], 1u);
          atomicOr(&g_stack_error, 1);
          ok = 0;
          break;
        }
        __nanosleep(32);
      }
    }
    __threadfence();
    gen = g + 1;
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// acc[b][0..3] = sum_r x_b(row k0 + r) * W[k0 + r][c0 .. c0 + 3] over R rows,
// the row values of x held by lane r (r < R) and broadcast by shuffles.
template <int B, int R>
__device__ __forceinline__ void gemv_item(const float* __restrict__ W, int ldw, int k0, int c0,
                                          const float (&xr)[B], float (&acc)[B][4]) {
  float4 w[R];
#pragma unroll
  for (int r = 0; r < R; ++r)
    w[r] = __ldg(reinterpret_cast<const float4*>(W + static_cast<int64_t>(k0 + r) * ldw + c0));
#pragma unroll
  for (int b = 0; b < B; ++b)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[b][j] = 0.f;
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const float xv = __shfl_sync(0xffffffffu, xr[b], r);
      acc[b][0] = fmaf(xv, w[r].x, acc[b][0]);
      acc[b][1] = fmaf(xv, w[r].y, acc[b][1]);
      acc[b][2] = fmaf(xv, w[r].z, acc[b][2]);
      acc[b][3] = fmaf(xv, w[r].w, acc[b][3]);
    }
  }
}

template <int B>
__global__ void __launch_bounds__(kThreads, 1) stack_fused_kernel(FusedParams p) {
  __shared__ float s_fq[kRowsB];
  __shared__ float s_fk[kRowsB];
  __shared__ __align__(16) float s_v[64];
  __shared__ float s_num[kWarps][64];
  __shared__ float s_den[kWarps];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int gwarp = blockIdx.x * kWarps + warp;
  const int nwarps = gridDim.x * kWarps;
  const int Dm = p.heads * 64;
  const int N = B * p.heads;                  // slots per layer
  const int64_t qkv_stride = static_cast<int64_t>(3) * B * Dm;
  unsigned gen = 0;

  for (int l = 0; l < p.L; ++l) {
    float* qkv = p.qkv + (l & 1) * qkv_stride;
    float* qkv_next = p.qkv + ((l + 1) & 1) * qkv_stride;
    // ---------------------------------------------------------------- A
    {
      // the other buffer (read by the previous layer's phase B) and the
      // readout sums (read by the previous layer's phase C) for this layer
      for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + tid; i < qkv_stride;
           i += static_cast<int64_t>(gridDim.x) * kThreads)
        qkv_next[i] = 0.f;
      for (int i = blockIdx.x * kThreads + tid; i < N * 65; i += gridDim.x * kThreads) {
        if (i < N * 64)
          p.num[i] = 0.f;
        else
          p.den[i - N * 64] = 0.f;
      }
      const float* W = p.Wqkv + static_cast<int64_t>(l) * Dm * 3 * Dm;
      const int ncb = 3 * Dm / 128;
      const int nitems = ncb * (Dm / kRowsA);
      for (int it = gwarp; it < nitems; it += nwarps) {
        const int cb = it % ncb, rb = it / ncb;
        const int c0 = cb * 128 + 4 * lane, k0 = rb * kRowsA;
        float xr[B];
#pragma unroll
        for (int b = 0; b < B; ++b)
          xr[b] = __ldcg(p.x + static_cast<int64_t>(b) * Dm + k0 + lane);
        float acc[B][4];
        gemv_item<B, kRowsA>(W, 3 * Dm, k0, c0, xr, acc);
        const int blk = c0 / Dm, col = c0 % Dm;   // q | k | v block and column (Dm % 4 == 0)
#pragma unroll
        for (int b = 0; b < B; ++b)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            red_add(qkv + (static_cast<int64_t>(blk) * B + b) * Dm + col + j, acc[b][j]);
      }
    }
    if (!grid_sync(p.bar, gen)) return;
    // ---------------------------------------------------------------- B
    {
      const int64_t slot_state = static_cast<int64_t>(384) * 64;
      for (int it = blockIdx.x; it < N * kParts; it += gridDim.x) {
        const int n = it / kParts, part = it % kParts;
        const int b = n / p.heads, h = n % p.heads;
        const int gh = l * p.heads + h;       // parameter row of the layer's head
        float* Sn = p.S + (static_cast<int64_t>(l) * N + n) * slot_state +
                    static_cast<int64_t>(part) * kRowsB * 64;
        float* zn = p.z + (static_cast<int64_t>(l) * N + n) * 384 + part * kRowsB;
        const int cgp = tid & 15, r0 = tid >> 4;
        float4 xs[kRowsB / 16];
#pragma unroll
        for (int i = 0; i < kRowsB / 16; ++i)
          xs[i] = reinterpret_cast<const float4*>(Sn)[(r0 + 16 * i) * 16 + cgp];
        const float zr = tid < kRowsB ? zn[tid] : 0.f;
        const float* qrow = qkv + static_cast<int64_t>(b) * Dm + h * 64;
        if (tid < 16) {
          const int a = part * 8 + (tid & 7);
          const float u = __ldcg((tid < 8 ? qrow : qrow + static_cast<int64_t>(B) * Dm) + a);
          const float ph = phase_mod_2pi(p.pos[n], p.phi[gh * 64 + a]);
          float ch[6];
          decm::feat_decode(u, p.gamma[gh], p.omega[gh * 64 + a], ph, ch);
          float* dst = (tid < 8 ? s_fq : s_fk) + 6 * (tid & 7);
#pragma unroll
          for (int c = 0; c < 6; ++c) dst[c] = ch[c];
        } else if (tid < 16 + 64) {
          s_v[tid - 16] = __ldcg(qrow + static_cast<int64_t>(2) * B * Dm + tid - 16);
        }
        __syncthreads();
        const float4 vv = reinterpret_cast<const float4*>(s_v)[cgp];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < kRowsB / 16; ++i) {
          const int r = r0 + 16 * i;
          const float pk = s_fk[r];
          float4 y = xs[i];
          y.x = fmaf(pk, vv.x, y.x);
          y.y = fmaf(pk, vv.y, y.y);
          y.z = fmaf(pk, vv.z, y.z);
          y.w = fmaf(pk, vv.w, y.w);
          reinterpret_cast<float4*>(Sn)[r * 16 + cgp] = y;
          const float pq = s_fq[r];
          acc.x = fmaf(pq, y.x, acc.x);
          acc.y = fmaf(pq, y.y, acc.y);
          acc.z = fmaf(pq, y.z, acc.z);
          acc.w = fmaf(pq, y.w, acc.w);
        }
        // lanes l and l + 16 of a warp hold the same column group
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, 16);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, 16);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, 16);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, 16);
        if (lane < 16) {
          s_num[warp][4 * cgp] = acc.x;
          s_num[warp][4 * cgp + 1] = acc.y;
          s_num[warp][4 * cgp + 2] = acc.z;
          s_num[warp][4 * cgp + 3] = acc.w;
        }
        float dn = 0.f;
        if (tid < kRowsB) {
          const float zz = zr + s_fk[tid];
          zn[tid] = zz;
          dn = s_fq[tid] * zz;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dn += __shfl_xor_sync(0xffffffffu, dn, off);
        if (lane == 0) s_den[warp] = dn;
        __syncthreads();
        if (tid < 64) {
          float s = 0.f;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) s += s_num[w][tid];
          red_add(p.num + static_cast<int64_t>(n) * 64 + tid, s);
        } else if (tid == 64) {
          float s = 0.f;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) s += s_den[w];
          red_add(p.den + n, s);
        }
        __syncthreads();   // the shared buffers are reused by the next item
      }
    }
    if (!grid_sync(p.bar, gen)) return;
    // ---------------------------------------------------------------- C
    {
      const float* W = p.Wo + static_cast<int64_t>(l) * Dm * Dm;
      const int ncb = Dm / 128;
      const int nitems = ncb * (Dm / kRowsC);
      for (int it = gwarp; it < nitems; it += nwarps) {
        const int cb = it % ncb, rb = it / ncb;
        const int c0 = cb * 128 + 4 * lane, k0 = rb * kRowsC;
        // o of rows k0 .. k0 + 15 (lane r < 16 holds row k0 + r; the rows lie in one head)
        float xr[B];
        const int kr = k0 + (lane & (kRowsC - 1));
        const int hh = kr / 64, e = kr % 64;
#pragma unroll
        for (int b = 0; b < B; ++b) {
          const int n = b * p.heads + hh;
          xr[b] = __ldcg(p.num + static_cast<int64_t>(n) * 64 + e) / (__ldcg(p.den + n) + p.eps);
        }
        float acc[B][4];
        gemv_item<B, kRowsC>(W, Dm, k0, c0, xr, acc);
#pragma unroll
        for (int b = 0; b < B; ++b)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            red_add(p.x + static_cast<int64_t>(b) * Dm + c0 + j, acc[b][j]);
      }
    }
    if (l + 1 < p.L && !grid_sync(p.bar, gen)) return;
  }
}

template <int B>
cudaError_t launch_fused(const FusedParams& fp, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stack_fused_kernel<B>, fp);
}

template <int B>
const void* fused_fn() {
  return reinterpret_cast<const void*>(stack_fused_kernel<B>);
}

using LaunchFn = cudaError_t (*)(const FusedParams&, int, cudaStream_t);
constexpr LaunchFn kLaunch[kMaxB] = {launch_fused<1>, launch_fused<2>, launch_fused<3>,
                                     launch_fused<4>, launch_fused<5>, launch_fused<6>,
                                     launch_fused<7>, launch_fused<8>};
using FnPtr = const void* (*)();
constexpr FnPtr kFn[kMaxB] = {fused_fn<1>, fused_fn<2>, fused_fn<3>, fused_fn<4>,
                              fused_fn<5>, fused_fn<6>, fused_fn<7>, fused_fn<8>};

// CTAs of the fused kernel: one per SM (0 when cooperative launches or one
// resident CTA per SM are not available).
int fused_grid(int B) {
  static int cached[kMaxB + 1] = {};
  if (cached[B] == 0) {
    int dev = 0, sms = 0, coop = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
        coop == 0)
      return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kFn[B - 1](), kThreads, 0) !=
            cudaSuccess ||
        per_sm < 1)
      return 0;
    cached[B] = sms;
  }
  return cached[B];
}

}  // namespace

size_t stack_workspace_bytes(int B, int heads, int d) {
  const size_t Dm = static_cast<size_t>(heads) * d;
  const size_t N = static_cast<size_t>(B) * heads;
  return (kBarWords + 2 * 3 * static_cast<size_t>(B) * Dm + N * 64 + N) * sizeof(float);
}

int stack_max_batch() { return kMaxB; }

int stack_read_and_clear_error(cudaStream_t st) {
  int h = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_stack_error, sizeof(int), 0, cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return -1;
  if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_stack_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                st) != cudaSuccess)
      return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  }
  return h;
}

cudaError_t stack_decode_launch(const StackArgs& a, cudaStream_t st) {
  if (a.B < 1 || a.B > kMaxB) return cudaErrorInvalidValue;
  const int grid = fused_grid(a.B);
  if (grid <= 0) return cudaErrorNotSupported;
  const int Dm = a.heads * 64;
  FusedParams fp{};
  fp.x = a.x;
  fp.Wqkv = a.Wqkv;
  fp.Wo = a.Wo;
  fp.S = a.S;
  fp.z = a.z;
  fp.gamma = a.gamma;
  fp.omega = a.omega;
  fp.phi = a.phi;
  fp.pos = a.pos;
  fp.L = a.L;
  fp.heads = a.heads;
  fp.eps = a.eps;
  float* ws = static_cast<float*>(a.workspace);
  fp.bar = reinterpret_cast<unsigned*>(ws);
  fp.qkv = ws + kBarWords;
  fp.num = fp.qkv + static_cast<int64_t>(2) * 3 * a.B * Dm;
  fp.den = fp.num + static_cast<int64_t>(a.B) * a.heads * 64;
  // the barrier words and the first layer's [q | k | v] buffer start at zero
  const cudaError_t e = cudaMemsetAsync(
      ws, 0, (kBarWords + static_cast<size_t>(3) * a.B * Dm) * sizeof(float), st);
  if (e != cudaSuccess) return e;
  return kLaunch[a.B - 1](fp, grid, st);
}

}  // namespace sanatan
