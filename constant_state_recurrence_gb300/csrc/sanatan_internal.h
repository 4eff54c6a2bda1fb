// Internal launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "sanatan.h"

namespace sanatan {

struct ChunkFwdArgs {
  const void* q;
  const void* k;
  const void* v;
  int in_dtype;
  const float* gamma;
  const float* omega;
  const float* phi;
  int B, H, T, d, dv;
  int64_t pos0;
  float eps;
  const float* S0;
  const float* z0;
  float* o;
  float* D;
  float* S_out;
  float* z_out;
  void* workspace;
  size_t workspace_bytes;
};

struct ChunkBwdArgs {
  ChunkFwdArgs f;
  const float* o;
  const float* Dn;
  const void* dO;
  int grad_dtype;
  void* dq;
  void* dk;
  void* dv;
  float* dgamma;
  float* domega;
  float* dphi;
  void* workspace;
  size_t workspace_bytes;
  const void* fwd_workspace;   // the forward's workspace (its per-segment sums) or null
  size_t fwd_workspace_bytes;
};

// Events recorded around the dominant kernel of a chunk_fwd / chunk_bwd call
// (bench instrumentation; null when unused).
struct ProfileEvents {
  cudaEvent_t start = nullptr;
  cudaEvent_t stop = nullptr;
};
ProfileEvents& profile_events();

cudaError_t featurize_launch(const void* u, int u_dtype, const float* gamma, const float* omega,
                             const float* phi, int B, int H, int T, int d, int64_t pos0,
                             void* out, int out_dtype, cudaStream_t st);

// phi = scale tanh(raw) (dphi == null) or dphi scale (1 - tanh^2(raw)).
cudaError_t rate_launch(const float* raw, const float* dphi, int n, float scale, float* out,
                        cudaStream_t st);

cudaError_t decode_step_launch(float* S, float* z, const float* q, const float* k,
                               const float* v, const float* gamma, const float* omega,
                               const float* phi, const int64_t* pos, int N, int G, float eps,
                               float* o, cudaStream_t st);

// Harmonic feature map (harmonics n = 1..N, N <= 3).
struct HarmonicFeatArgs {
  const void* u;
  int u_dtype;
  const float* gamma;
  const float* omega;
  const float* phi;
  int B, H, T;
  int64_t pos0;
  int harmonics;
  void* out;
  int out_dtype;
};
cudaError_t featurize_harmonic_launch(const HarmonicFeatArgs& a, cudaStream_t st);
// f32 chunked forward with the harmonic map (N <= 3; bf16 or f32 loads).
cudaError_t chunk_fwd_harmonic_launch(const ChunkFwdArgs& a, int harmonics, cudaStream_t st);
// Its backward (N <= 3); the workspace holds dN and dD (none for N = 1).
size_t chunk_bwd_harmonic_workspace_bytes(int B, int H, int T, int harmonics);
cudaError_t chunk_bwd_harmonic_launch(const ChunkBwdArgs& a, int harmonics, cudaStream_t st);
cudaError_t decode_harmonic_launch(float* S, float* z, const float* q, const float* k,
                                   const float* v, const float* gamma, const float* omega,
                                   const float* phi, const int64_t* pos, int N, int G, float eps,
                                   int harmonics, float* o, cudaStream_t st);

// One token through L attention layers (stack.cu): one cooperative launch.
struct StackArgs {
  float* x;              // [B, heads * 64], updated in place
  const float* Wqkv;     // [L, heads * 64, 3 * heads * 64]
  const float* Wo;       // [L, heads * 64, heads * 64]
  float* S;              // [L, B * heads, 384, 64]
  float* z;              // [L, B * heads, 384]
  const float* gamma;    // [L, heads]
  const float* omega;    // [L, heads, 64]
  const float* phi;      // [L, heads, 64]
  const int64_t* pos;    // [B * heads]
  int B, L, heads;
  float eps;
  void* workspace;       // stack_workspace_bytes
};
size_t stack_workspace_bytes(int B, int heads, int d);
int stack_max_batch();
cudaError_t stack_decode_launch(const StackArgs& a, cudaStream_t st);
int stack_read_and_clear_error(cudaStream_t st);

size_t chunk_fwd_simt_smem_bytes();
size_t chunk_bwd_simt_smem_bytes();
cudaError_t chunk_bwd_simt_launch(const ChunkBwdArgs& a, cudaStream_t st);
cudaError_t chunk_fwd_simt_launch(const ChunkFwdArgs& a, cudaStream_t st);

}  // namespace sanatan

namespace sanatan {
int tc_segments(int B, int H, int T);
size_t chunk_fwd_tc_workspace_bytes(int B, int H, int T);
cudaError_t chunk_fwd_tc_launch(const ChunkFwdArgs& a, cudaStream_t st);
int tc_read_and_clear_error(cudaStream_t st);
// One CTA whose bounded wait on an mbarrier nobody arrives at (unless
// `arrive`) gives up after timeout_ns and records a timeout.
cudaError_t tc_timeout_probe_launch(uint64_t timeout_ns, int arrive, cudaStream_t st);

// One causal (or, reversed, anti-causal) attention on the tensor-core kernel,
// bf16 q, k, v of shape [B, H, T, 64].  `extra` replaces the ones column of
// [V | 1] (the denominator) by a per-token value; `deltas` is the workspace of
// per-segment state sums, B * H * tc_segments * 321 * 80 floats.
struct TcJob {
  const void* q = nullptr;
  const void* k = nullptr;
  const void* v = nullptr;
  const float* extra = nullptr;
  const float* gamma = nullptr;
  const float* omega = nullptr;
  const float* phi = nullptr;
  int B = 0, H = 0, T = 0;
  int64_t pos0 = 0;
  float eps = 0.f;
  const float* S0 = nullptr;
  const float* z0 = nullptr;
  void* o = nullptr;        // f32 or (out_bf16) bf16 [B, H, T, 64]
  float* Dn = nullptr;
  float* S_out = nullptr;
  float* z_out = nullptr;
  int reverse = 0;          // row u is processed at position T-1-u
  int normalize = 1;        // 0: write the numerator only
  int out_bf16 = 0;
  float* deltas = nullptr;
  int deltas_ready = 0;     // the state-only pass has already filled `deltas`
  int record_events = 1;    // bracket the main launch with the profile events
  int nseg = 0;             // segments per sequence (0: tc_segments)
};
// State-only pass: the sums of every segment but the last into job.deltas.
cudaError_t tc_state_pass(const TcJob& job, cudaStream_t st);
// The attention itself (running the state-only pass first unless deltas_ready).
cudaError_t tc_attention(const TcJob& job, cudaStream_t st);

size_t chunk_bwd_tc_workspace_bytes(int B, int H, int T);
// Segments that a workspace of `bytes` holds (at most tc_segments; 1 needs none).
int tc_segments_fit(int B, int H, int T, size_t bytes);
int chunk_fwd_checked(const void* q, const void* k, const void* v, int in_dtype,
                      const float* gamma, const float* omega, const float* phi, int B, int H,
                      int T, int d, int dv, int64_t pos0, float eps, const float* S0,
                      const float* z0, float* o, float* D, float* S_out, float* z_out,
                      void* workspace, size_t workspace_bytes, void* stream, bool fewer_segments);
cudaError_t chunk_bwd_tc_launch(const ChunkBwdArgs& a, cudaStream_t st);
int bwd_tc_read_and_clear_error(cudaStream_t st);

// Power-sharpened causal attention (bf16 q, k, v [B, H, T, 64], integer p).
struct PowFwdArgs {
  const void* q = nullptr;
  const void* k = nullptr;
  const void* v = nullptr;
  const float* gamma = nullptr;
  const float* omega = nullptr;
  const float* phi = nullptr;
  int B = 0, H = 0, T = 0;
  int64_t pos0 = 0;
  int p = 1;
  float eps = 0.f;
  float* o = nullptr;
  float* D = nullptr;
  void* workspace = nullptr;   // pow_fwd_tc_workspace_bytes
};
size_t pow_fwd_tc_workspace_bytes(int B, int H, int T);
cudaError_t pow_fwd_tc_launch(const PowFwdArgs& a, cudaStream_t st);
// The four- (channels = 4) or three-channel (channels = 3, with `shift`) map in
// the same kernels; p in {1, 2, 4}.
cudaError_t ablation_fwd_tc_launch(const PowFwdArgs& a, int channels, float shift,
                                   cudaStream_t st);
// The preparation kernel alone (features and [V | 1 | 0] into a.workspace).
cudaError_t pow_prep_launch(const PowFwdArgs& a, cudaStream_t st);

// Gradients of the power-sharpened attention.
struct PowBwdArgs {
  PowFwdArgs f;               // q, k, v, params, sizes, p, eps; f.workspace = the whole workspace
  const float* o = nullptr;   // [B, H, T, 64] f32, the forward's output
  const float* D = nullptr;   // [B, H, T] f32, the forward's denominator (without eps)
  const void* dO = nullptr;   // [B, H, T, 64], grad_dtype
  int grad_dtype = 0;
  void* dq = nullptr;         // bf16 [B, H, T, 64]
  void* dk = nullptr;
  void* dv = nullptr;
  float* dgamma = nullptr;    // [H], overwritten
  float* domega = nullptr;    // [H, 64], overwritten
  float* dphi = nullptr;      // [H, 64], overwritten (may be null)
};
size_t pow_bwd_tc_workspace_bytes(int B, int H, int T);
cudaError_t pow_bwd_tc_launch(const PowBwdArgs& a, cudaStream_t st);
int pow_bwd_tc_read_and_clear_error(cudaStream_t st);
int pow_tc_read_and_clear_error(cudaStream_t st);
}  // namespace sanatan
