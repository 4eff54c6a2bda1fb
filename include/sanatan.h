/*
 * sanatan.h -- C ABI of libsanatan.so: SANATAN p=1 root-parity gated angular
 * attention on NVIDIA GB300 (sm_103a).
 *
 * The method is that of "SANATAN: Root-Parity Gated Angular Attention with an
 * Exact Constant-State Recurrent Form" (B. Patel), as summarised by its reading
 * notes (cited as "Notes") and the author's post.  Each query/key component u
 * of a head becomes an angle theta = pi u / (1 + |u|) (Notes §2.2, eq. (2)); a
 * soft root label r = tanh(gamma (cos(theta+omega) - sin(theta+omega))) is
 * taken from that un-rotated angle (eq. (3)); the angle is rotated by
 * t * phi_a (eq. (4)); the six channels
 *     Phi_a = [1, cos theta_rot, sin theta_rot, r, r cos theta_rot, r sin theta_rot]
 * are concatenated over the d dimensions (eq. (6), Notes §2.3).  Attention at
 * p = 1 is causal and normalised (eq. (9), Notes §2.7):
 *     S_t = S_{t-1} + Phi(k_t) v_t^T,   z_t = z_{t-1} + Phi(k_t),
 *     o_t = Phi(q_t)^T S_t / (Phi(q_t)^T z_t + eps),
 * the update preceding the read (the mask includes the current token).
 *
 * Conventions shared by every call
 *  - Every pointer is DEVICE memory owned by the caller, unless stated.
 *    The library allocates no device memory and keeps no state between calls
 *    except cached device attributes.
 *  - Tensors are dense and row-major (C order) with the shapes given below;
 *    pointers must be 16-byte aligned (SANATAN_ERR_INVALID otherwise).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  No call synchronises the device; a status of SANATAN_OK means
 *    the launches were enqueued without a launch error.
 *  - Feature index inside the 6d axis is 6*a + c, channel order as above.
 *  - Positions: token i of a sequence sits at t = pos0 + i.
 *  - eps is added to the denominator in raw score units (default 0).
 *  - gamma [H], omega [H, d], phi [H, d] are float32; omega is shared by q and k
 *    of a head; phi is the per-dimension rotation rate.
 *  - d = dv = 64 is the supported head size (SANATAN_ERR_UNSUPPORTED otherwise).
 *  - Arguments are validated on the host before anything is launched; on an
 *    error status nothing has been enqueued (except SANATAN_ERR_CUDA, which
 *    reports a failed launch).
 */
#ifndef SANATAN_H_
#define SANATAN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SANATAN_API __attribute__((visibility("default")))
#else
#define SANATAN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum sanatan_status {
  SANATAN_OK = 0,
  SANATAN_ERR_INVALID = 1,     /* null/misaligned pointer, negative size, bad enum */
  SANATAN_ERR_UNSUPPORTED = 2, /* a shape or dtype this build does not handle     */
  SANATAN_ERR_CUDA = 3,        /* a CUDA runtime error (launch or attribute query) */
  SANATAN_ERR_ARCH = 4,        /* the current device is not sm_103 (GB300)          */
  SANATAN_ERR_TIMEOUT = 5      /* a device-side bounded wait gave up                */
};

/* Element types of q, k, v (and of dq, dk, dv, dO where stated). */
enum sanatan_dtype { SANATAN_F32 = 0, SANATAN_BF16 = 1 };

/* Human-readable text of a status code (static storage, never NULL). */
SANATAN_API const char* sanatan_status_string(int status);

/* ABI version of this library (increments when a signature changes). */
SANATAN_API int sanatan_abi_version(void);

/* Bytes of recurrent state of one sequence with `layers` x `heads` heads:
 * per head S (6d x dv) and z (6d) float32 (Notes §4.5, paper §4.4:
 * 12 x 12 x (6*64*64 + 6*64) x 4 = 14,376,960 bytes). Host-only arithmetic. */
SANATAN_API size_t sanatan_state_bytes(int layers, int heads, int d, int dv);

/*
 * sanatan_featurize -- the feature map Phi of eqs. (2)-(6) (Notes §2.2-§2.3).
 *   u       [B, H, T, d]   u_dtype (SANATAN_F32 or SANATAN_BF16)
 *   gamma   [H] f32, omega [H, d] f32, phi [H, d] f32
 *   out     [B, H, T, 6d]  out_dtype; out[..., 6a + c] is channel c of dim a
 * Float32 output is computed with correctly rounded division and libm-grade
 * sin/cos/tanh; bf16 output is the float32 value rounded to nearest even.
 */
SANATAN_API int sanatan_featurize(const void* u, int u_dtype, const float* gamma, const float* omega,
                      const float* phi, int B, int H, int T, int d, int64_t pos0, void* out,
                      int out_dtype, void* stream);

/*
 * sanatan_rate_from_raw -- the rotation rate of eq. (4) from its unconstrained
 * parameter, as the notes give it (§2.2): phi = scale * tanh(lambda_raw) with
 * scale = 0.01 on the pages (any scale is accepted).  lambda_raw and phi are
 * n float32 values on the device (e.g. [H, d]); phi may be passed to every
 * call that takes phi.  SANATAN_ERR_INVALID for n < 0 or a null/misaligned
 * pointer (n = 0 does nothing).
 * sanatan_rate_from_raw_bwd -- the gradient of the same map:
 * dlambda_raw = dphi * scale * (1 - tanh^2(lambda_raw)), e.g. for the dphi of
 * sanatan_chunk_bwd.
 */
SANATAN_API int sanatan_rate_from_raw(const float* lambda_raw, int n, float scale, float* phi,
                                      void* stream);
SANATAN_API int sanatan_rate_from_raw_bwd(const float* lambda_raw, const float* dphi, int n,
                                          float scale, float* dlambda_raw, void* stream);

/*
 * sanatan_eps_raw -- the raw-score eps that reproduces a parallel form which
 * divides scores by c before adding eps (notes §2.7: eps_raw = c * eps):
 * convention 0 takes the authors' parallel code's c = 4d + 1e-6, convention 1
 * the recurrence notebook's approximation c = 4d * 1e-6.  Host-only
 * arithmetic; returns -1 for d <= 0 or another convention.
 */
SANATAN_API float sanatan_eps_raw(float eps, int d, int convention);

/*
 * sanatan_chunk_fwd -- causal normalised attention at p = 1 over whole
 * sequences (eq. (9) evaluated chunk-parallel; the exact re-association of the
 * sums in Notes §2.7), optionally continuing from a state (S0, z0).
 *   q, k    [B, H, T, d]   in_dtype;   v [B, H, T, dv] in_dtype
 *   S0      [B, H, 6d, dv] f32 or NULL (zero state); z0 [B, H, 6d] f32 or NULL
 *           (S0 and z0 are both NULL or both non-NULL)
 *   o       [B, H, T, dv]  f32 output
 *   D       [B, H, T]      f32 output or NULL: the denominator Phi(q_t)^T z_t
 *           (without eps), kept for the backward
 *   S_out   [B, H, 6d, dv] f32 output or NULL: the state after token T-1
 *   z_out   [B, H, 6d]     f32 output or NULL (both or neither with S_out)
 *   workspace / workspace_bytes: device scratch of at least
 *           sanatan_chunk_fwd_workspace_size(...) bytes (may be NULL if that
 *           size is 0); its contents on entry do not matter.
 * bf16 inputs run on the tensor cores (bf16 operands, f32 accumulation);
 * f32 inputs run an all-f32 CUDA-core path.  T = 0 is valid and does nothing
 * but copy (S0, z0) (or zeros) to (S_out, z_out).
 */
SANATAN_API size_t sanatan_chunk_fwd_workspace_size(int B, int H, int T, int d, int dv, int in_dtype);
/* How sanatan_chunk_fwd splits a problem: *segments = segments per sequence
 * (the long-sequence split of the tensor-core path), *launches = kernels one
 * call enqueues.  Host-only arithmetic (reads the current device's SM count). */
SANATAN_API int sanatan_chunk_fwd_plan(int B, int H, int T, int in_dtype, int has_initial_state,
                                       int* segments, int* launches);
SANATAN_API int sanatan_chunk_fwd(const void* q, const void* k, const void* v, int in_dtype,
                      const float* gamma, const float* omega, const float* phi, int B, int H,
                      int T, int d, int dv, int64_t pos0, float eps, const float* S0,
                      const float* z0, float* o, float* D, float* S_out, float* z_out,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * sanatan_chunk_fwd_noalloc -- sanatan_chunk_fwd for bf16 inputs that takes no
 * workspace and allocates nothing.  The paper has no counterpart: this entry
 * exists for callers that cannot hand the library device scratch memory, e.g.
 * a plugin that only receives its input and output buffers from a host
 * framework, or code running where cudaMalloc is off limits because it
 * implicitly synchronises the device or because a pool owns all device memory.
 *   Arguments and results are those of sanatan_chunk_fwd with in_dtype =
 *   SANATAN_BF16 and without the workspace pair.
 *   Scratch: a fixed array inside the library, 16 MiB per device
 *   (sanatan_chunk_fwd_noalloc_max_scratch_bytes()), held by every GPU that
 *   loads the library until the process exits.  It holds the per-segment
 *   state sums of the long-sequence split: a problem whose preferred split
 *   (sanatan_chunk_fwd_workspace_size) needs more than 16 MiB runs with as
 *   many segments per sequence as the array holds (one segment needs no
 *   scratch), so every problem size sanatan_chunk_fwd accepts runs here too,
 *   with the same results up to rounding; only the split, and so the speed,
 *   can differ.  SANATAN_ERR_UNSUPPORTED is returned only if a split would
 *   ever need more than the array (it cannot with this build's split rule).
 *   The first call on a device looks up the array's device address (no
 *   allocation); make that first call before any stream capture.
 *   Calls share the array: two calls whose kernels overlap on the GPU (other
 *   streams, other threads) race on it and give undefined results.  The
 *   kernels overwrite every scratch byte before reading it, so nothing needs
 *   clearing between calls.
 */
SANATAN_API size_t sanatan_chunk_fwd_noalloc_max_scratch_bytes(void);
SANATAN_API int sanatan_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                          const float* gamma, const float* omega,
                                          const float* phi, int B, int H, int T, int d, int dv,
                                          int64_t pos0, float eps, const float* S0,
                                          const float* z0, float* o, float* D, float* S_out,
                                          float* z_out, void* stream);

/*
 * sanatan_chunk_bwd -- gradients of sum(o * dO) for sanatan_chunk_fwd.
 * The chain rule through eqs. (2)-(4), (6), (9); the pages give no backward.
 *   q, k, v, gamma, omega, phi, sizes, pos0, eps, S0, z0: as for the forward
 *   o       [B, H, T, dv] f32 and D [B, H, T] f32: the forward's outputs
 *   dO      [B, H, T, dv] in grad_dtype (SANATAN_F32 or SANATAN_BF16)
 *   dq, dk  [B, H, T, d]  in_dtype outputs;  dv_out [B, H, T, dv] in_dtype
 *   dgamma  [H] f32 output, domega [H, d] f32 output (overwritten, summed over
 *           the batch and both q and k), dphi [H, d] f32 output or NULL
 *   workspace: at least sanatan_chunk_bwd_workspace_size(...) bytes.
 *   fwd_workspace / fwd_workspace_bytes: NULL / 0, or the workspace of the
 *           sanatan_chunk_fwd call that produced o and D from these same q, k,
 *           v, gamma, omega, phi and pos0, unchanged since.  On the bf16 path,
 *           when that workspace holds the forward's per-segment state sums for
 *           the backward's own split (the forward's preferred workspace size
 *           or more), the backward reuses them instead of recomputing them
 *           (one launch fewer); otherwise it is ignored.  Passing a workspace
 *           of another call gives wrong gradients.
 */
SANATAN_API size_t sanatan_chunk_bwd_workspace_size(int B, int H, int T, int d, int dv, int in_dtype);
SANATAN_API int sanatan_chunk_bwd(const void* q, const void* k, const void* v, int in_dtype,
                      const float* gamma, const float* omega, const float* phi, int B, int H,
                      int T, int d, int dv, int64_t pos0, float eps, const float* S0,
                      const float* z0, const float* o, const float* D, const void* dO,
                      int grad_dtype, void* dq, void* dk, void* dv_out, float* dgamma,
                      float* domega, float* dphi, void* workspace, size_t workspace_bytes,
                      const void* fwd_workspace, size_t fwd_workspace_bytes, void* stream);

/*
 * sanatan_power_fwd -- power-sharpened causal attention, eq. (8) (Notes §2.6),
 * at a positive integer power p, in the parallel (quadratic) form the paper
 * trains with; for p > 1 it has no constant-size state:
 *     a_tj = (s_tj / 4d)^p / (sum_{l<=t} (s_tl / 4d)^p + eps),
 *     o_t  = sum_{j<=t} a_tj v_j,      s_tj = Phi(q_t) . Phi(k_j).
 * At p = 1 it equals sanatan_chunk_fwd with eps multiplied by 4d.
 *   q, k    [B, H, T, d]  bf16;  v [B, H, T, dv] bf16
 *   p       1 <= p <= 8 (SANATAN_ERR_INVALID below 1, SANATAN_ERR_UNSUPPORTED above 8)
 *   o       [B, H, T, dv] f32 output
 *   D       [B, H, T] f32 output or NULL: sum_{l<=t} (s_tl / 4d)^p, without eps
 *   workspace / workspace_bytes: device scratch of at least
 *           sanatan_power_fwd_workspace_size(...) bytes (about 1.4 KB per
 *           token, rounded up to whole 128-token chunks): the bf16 features
 *           Phi(q), Phi(k) and v laid out for the tensor cores; its contents on
 *           entry do not matter.
 * Scores, the power and the denominator are float32; features and values
 * enter the tensor cores as bf16, the weights (s/4d)^p as a bf16 pair (hi +
 * lo), and the tensor core sums the same weights for the denominator.
 * T = 0 or B * H = 0 does nothing.  Errors: SANATAN_ERR_INVALID for a null
 * or misaligned pointer (D may be NULL) or a workspace smaller than the size
 * above; SANATAN_ERR_UNSUPPORTED for d or dv other than 64 or more than 2^30
 * (sequence, 128-token chunk) pairs.
 */
SANATAN_API size_t sanatan_power_fwd_workspace_size(int B, int H, int T, int d, int dv);
SANATAN_API int sanatan_power_fwd(const void* q, const void* k, const void* v, const float* gamma,
                                  const float* omega, const float* phi, int B, int H, int T, int d,
                                  int dv, int64_t pos0, int p, float eps, float* o, float* D,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * sanatan_ablation_fwd -- the power-sharpened causal attention of
 * sanatan_power_fwd with one of the two ablation feature maps of the notes in
 * place of the six-channel map (same squash, soft root from the un-rotated
 * angle, and rotation):
 *   channels = 4: Phi4_a = [1, r, r cos th_rot, r sin th_rot] (Notes §2.5).  The
 *       per-dimension kernel 1 + r_q r_k (1 + cos dth) can be negative, and the
 *       total score is clipped at zero before the power:
 *       w_tj = (max(s_tj, 0) / 3d)^p.
 *   channels = 3: Phi3_a = [1, cos th_rot, sin th_rot] (Notes §4.4), so
 *       s_tj = d + sum_a cos dth_a in [0, 2d]; `shift` is added to every score
 *       first (the printed ablation adds d; shift = 0 is the fair ablation the
 *       notes ask for): w_tj = ((s_tj + shift) / (2d + shift))^p.
 *   o_t = sum_{j<=t} w_tj v_j / (sum_{j<=t} w_tj + eps);  D_t = sum_{j<=t} w_tj.
 *   p in {1, 2, 4}.  Other arguments, layouts, the workspace
 *   (sanatan_power_fwd_workspace_size) and errors as for sanatan_power_fwd;
 *   SANATAN_ERR_INVALID for channels other than 3 or 4, a negative shift or a
 *   nonzero shift with channels = 4; SANATAN_ERR_UNSUPPORTED for another p.
 */
SANATAN_API int sanatan_ablation_fwd(const void* q, const void* k, const void* v,
                                     const float* gamma, const float* omega, const float* phi,
                                     int B, int H, int T, int d, int dv, int64_t pos0, int p,
                                     int channels, float shift, float eps, float* o, float* D,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * sanatan_power_bwd -- gradients of sum(o * dO) for sanatan_power_fwd (the
 * chain rule through eq. (8) and the feature map; the pages give no backward).
 *   q, k, v, gamma, omega, phi, sizes, pos0, p, eps: as for the forward
 *   o [B, H, T, dv] f32 and D [B, H, T] f32: the forward's outputs
 *   dO [B, H, T, dv] in grad_dtype (SANATAN_F32 or SANATAN_BF16)
 *   dq, dk [B, H, T, d] bf16 outputs; dv_out [B, H, T, dv] bf16 output
 *   dgamma [H] f32, domega [H, d] f32 outputs (overwritten, summed over the
 *   batch and both q and k); dphi [H, d] f32 output or NULL
 *   workspace: at least sanatan_power_bwd_workspace_size(...) bytes.
 * Errors as for sanatan_power_fwd; grad_dtype outside the enum is INVALID.
 */
SANATAN_API size_t sanatan_power_bwd_workspace_size(int B, int H, int T, int d, int dv);
SANATAN_API int sanatan_power_bwd(const void* q, const void* k, const void* v, const float* gamma,
                                  const float* omega, const float* phi, int B, int H, int T, int d,
                                  int dv, int64_t pos0, int p, float eps, const float* o,
                                  const float* D, const void* dO, int grad_dtype, void* dq,
                                  void* dk, void* dv_out, float* dgamma, float* domega,
                                  float* dphi, void* workspace, size_t workspace_bytes,
                                  void* stream);

/*
 * sanatan_set_profile_events -- instrumentation for benchmarks.  When both
 * are non-NULL, the calling thread's subsequent sanatan_chunk_fwd,
 * sanatan_chunk_bwd and sanatan_power_fwd calls record `start` (a cudaEvent_t) on their stream just
 * before their dominant kernel launch and `stop` just after it, so the caller
 * can time that kernel alone.  Pass NULL, NULL to turn it off.  Thread-local;
 * the events stay owned by the caller.
 */
SANATAN_API int sanatan_set_profile_events(void* start, void* stop);

/*
 * sanatan_device_status -- synchronises `stream`, then reports whether any
 * kernel of this library gave up a bounded device-side wait since the last
 * call (SANATAN_ERR_TIMEOUT; the flag is cleared) or not (SANATAN_OK).  The
 * tensor-core kernels never spin without a time limit: a lost hand-off makes
 * them skip their remaining waits and return, with undefined outputs.
 */
SANATAN_API int sanatan_device_status(void* stream);

/*
 * Harmonic feature map (the notes' Appendix B, "附录 B 的频谱展望"): harmonics
 * cos(n th), sin(n th), n = 1..N, added to the angle block; at p = 1 the
 * attention stays an explicit feature-map attention with a constant-size state
 * of F_N = 2(2N + 1) d features (N = 1: the six-channel map).  Per dimension a
 * the channels are [A, r A], A = [1, cos th, sin th, ..., cos N th, sin N th]
 * with th the rotated angle and r the root of the un-rotated one; channel
 * l (2N + 1) + m of dimension a sits at a * 2(2N + 1) + l (2N + 1) + m.  The
 * kernel is sum_a (1 + r_q r_k)(1 + sum_n cos(n dtheta_a)).  These calls run in
 * float32 on the CUDA cores.
 *
 * sanatan_state_bytes_harmonic -- bytes of S (F_N x dv) and z (F_N) float32 of
 *   layers x heads heads (host arithmetic; 0 for harmonics < 1).
 * sanatan_featurize_harmonic -- Phi_N(u) [B, H, T, F_N] in out_dtype for u
 *   [B, H, T, d]; harmonics 1..3 (SANATAN_ERR_UNSUPPORTED above 3).
 * sanatan_chunk_fwd_harmonic -- the causal normalised attention of
 *   sanatan_chunk_fwd with Phi_N (arguments, layouts and outputs as there with
 *   6d replaced by F_N; no workspace); q, k, v f32 or bf16 (converted to f32);
 *   harmonics 1..3 (N >= 2: a cluster of eight CTAs per sequence, each
 *   holding the state rows of eight dimensions in registers).
 * sanatan_chunk_bwd_harmonic -- gradients of sum(o * dO) for
 *   sanatan_chunk_fwd_harmonic (the chain rule of the six-channel backward
 *   with Phi_N; the pages give no backward).  Arguments, layouts and outputs
 *   as sanatan_chunk_bwd (dq, dk, dv_out in in_dtype; dgamma [H], domega
 *   [H, d] and dphi [H, d] (or NULL) float32, overwritten, summed over the
 *   batch and both q and k), without the forward-workspace pair; harmonics
 *   1..3.  workspace: at least sanatan_chunk_bwd_harmonic_workspace_size(...)
 *   bytes (65 floats per token-head: dN = dO / (D + eps) and
 *   dD = -(dO . o) / (D + eps); 0 for harmonics = 1, which runs the six-channel
 *   float32 backward); its contents on entry do not matter.  Arithmetic in
 *   float32 on the CUDA cores; float atomics make dgamma, domega, dphi vary in
 *   their last bits between runs.  Errors as sanatan_chunk_bwd, and
 *   SANATAN_ERR_INVALID for a workspace smaller than the size above.
 * sanatan_decode_step_harmonic -- one token of the recurrence with Phi_N for N
 *   slots, as sanatan_decode_step with S [N, F_N, dv] and z [N, F_N];
 *   harmonics 1..3.
 */
SANATAN_API size_t sanatan_state_bytes_harmonic(int layers, int heads, int d, int dv,
                                                int harmonics);
SANATAN_API int sanatan_featurize_harmonic(const void* u, int u_dtype, const float* gamma,
                                           const float* omega, const float* phi, int B, int H,
                                           int T, int d, int64_t pos0, int harmonics, void* out,
                                           int out_dtype, void* stream);
SANATAN_API int sanatan_chunk_fwd_harmonic(const void* q, const void* k, const void* v,
                                           int in_dtype, const float* gamma, const float* omega,
                                           const float* phi, int B, int H, int T, int d, int dv,
                                           int64_t pos0, int harmonics, float eps, const float* S0,
                                           const float* z0, float* o, float* D, float* S_out,
                                           float* z_out, void* stream);
SANATAN_API size_t sanatan_chunk_bwd_harmonic_workspace_size(int B, int H, int T, int d, int dv,
                                                             int harmonics);
SANATAN_API int sanatan_chunk_bwd_harmonic(const void* q, const void* k, const void* v,
                                           int in_dtype, const float* gamma, const float* omega,
                                           const float* phi, int B, int H, int T, int d, int dv,
                                           int64_t pos0, int harmonics, float eps,
                                           const float* S0, const float* z0, const float* o,
                                           const float* D, const void* dO, int grad_dtype,
                                           void* dq, void* dk, void* dv_out, float* dgamma,
                                           float* domega, float* dphi, void* workspace,
                                           size_t workspace_bytes, void* stream);
SANATAN_API int sanatan_decode_step_harmonic(float* S, float* z, const float* q, const float* k,
                                             const float* v, const float* gamma,
                                             const float* omega, const float* phi,
                                             const int64_t* pos, int N, int G, int d, int dv,
                                             int harmonics, float eps, float* o, void* stream);

/*
 * sanatan_stack_decode_step -- one decode token through L attention layers of
 * `heads` heads (the notes §2.7: the whole-model recurrence updates the layers'
 * states in order, each layer with its own weights, at the same positions;
 * §3.1: 12 layers x 12 heads x d = 64).  The attention path only, float32:
 * per layer l
 *     [q | k | v] = x Wqkv[l],  o = sanatan_decode_step of the layer's slots,
 *     x <- x + o Wo[l].
 *   x     [B, heads * d] f32, read and written (the token's input, then output)
 *   Wqkv  [L, heads * d, 3 * heads * d] f32 (columns: q | k | v, head-major)
 *   Wo    [L, heads * d, heads * d] f32
 *   S     [L, B * heads, 6d, d] f32 and z [L, B * heads, 6d] f32, updated in
 *         place (slot b * heads + h of layer l)
 *   gamma [L, heads], omega, phi [L, heads, d] f32
 *   pos   [B * heads] int64: the position of the token, per slot
 *   workspace: sanatan_stack_decode_workspace_size(B, heads, d) bytes.
 * B <= 8 and heads * d a multiple of 128 (SANATAN_ERR_UNSUPPORTED otherwise).
 * The projections accumulate with float atomics, so results can differ in the
 * last bits from run to run.
 */
SANATAN_API size_t sanatan_stack_decode_workspace_size(int B, int heads, int d);
SANATAN_API int sanatan_stack_decode_step(float* x, const float* Wqkv, const float* Wo, float* S,
                                          float* z, const float* gamma, const float* omega,
                                          const float* phi, const int64_t* pos, int B, int L,
                                          int heads, int d, float eps, void* workspace,
                                          size_t workspace_bytes, void* stream);

/*
 * sanatan_selftest_wait_timeout -- failure-detection self-test (the paper has
 * no counterpart).  Enqueues one small kernel whose thread waits, with the
 * same bounded mbarrier wait the tensor-core kernels use, on a barrier that
 * nothing arrives at (arrive = 0) or that another thread completes (arrive =
 * 1).  After timeout_ns (1e3 <= timeout_ns <= 1e9, SANATAN_ERR_INVALID
 * otherwise) the wait gives up and records a timeout in the library's device
 * error word, so the next sanatan_device_status returns SANATAN_ERR_TIMEOUT;
 * with arrive = 1 nothing is recorded.  The probe touches no caller memory and
 * leaves the CUDA context usable.
 */
SANATAN_API int sanatan_selftest_wait_timeout(uint64_t timeout_ns, int arrive, void* stream);

/*
 * sanatan_decode_step -- one token of the constant-state recurrence of eq. (9)
 * (Notes §2.7) for N independent state slots, updating the state IN PLACE.
 *   S       [N, 6d, dv] f32, read and written;  z [N, 6d] f32, read and written
 *   q, k    [N, d] f32;  v [N, dv] f32
 *   gamma [G] f32, omega [G, d] f32, phi [G, d] f32: slot n uses row g = n % G
 *           (G = layers x heads when slots are ordered sequence-major)
 *   pos     [N] int64: the position t of this token in each slot's sequence
 *   o       [N, dv] f32 output
 * The state written is S + Phi(k) v^T, z + Phi(k); the read uses the updated
 * state.
 */
SANATAN_API int sanatan_decode_step(float* S, float* z, const float* q, const float* k, const float* v,
                        const float* gamma, const float* omega, const float* phi,
                        const int64_t* pos, int N, int G, int d, int dv, float eps, float* o,
                        void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SANATAN_H_ */
