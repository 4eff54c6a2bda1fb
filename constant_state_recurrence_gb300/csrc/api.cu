// C ABI of libsanatan.so: host-side validation and dispatch (see sanatan.h).
#include <cstdint>
#include <cstring>

#include "sanatan_internal.h"

namespace {

using namespace sanatan;

constexpr int kAbiVersion = 2;
constexpr int kMaxPower = 8;   // largest p of sanatan_power_fwd

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }
bool ok_nullable(const void* p) { return p == nullptr || aligned16(p); }
bool ok_dtype(int t) { return t == SANATAN_F32 || t == SANATAN_BF16; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? SANATAN_OK : SANATAN_ERR_CUDA; }

// The kernels are built for sm_103a only; refuse any other device before a
// launch could fail with "no kernel image".
int check_arch() {
  static int cached[64];  // 0 unknown, 1 ok, 2 wrong arch
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SANATAN_ERR_CUDA;
  if (dev >= 0 && dev < 64 && cached[dev] != 0) return cached[dev] == 1 ? SANATAN_OK : SANATAN_ERR_ARCH;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return SANATAN_ERR_CUDA;
  const bool ok = (major == 10 && minor == 3);
  if (dev >= 0 && dev < 64) cached[dev] = ok ? 1 : 2;
  return ok ? SANATAN_OK : SANATAN_ERR_ARCH;
}

int check_sizes(int B, int H, int T, int d, int dv) {
  if (B < 0 || H < 0 || T < 0 || d < 0 || dv < 0) return SANATAN_ERR_INVALID;
  if (d != 64 || dv != 64) return SANATAN_ERR_UNSUPPORTED;
  // Element counts index with 64-bit arithmetic; CTA counts must fit a grid.
  if (static_cast<int64_t>(B) * H > (1LL << 31) - 1) return SANATAN_ERR_UNSUPPORTED;
  return SANATAN_OK;
}

int check_params(const float* gamma, const float* omega, const float* phi) {
  if (!ok_ptr(gamma) || !ok_ptr(omega) || !ok_ptr(phi)) return SANATAN_ERR_INVALID;
  return SANATAN_OK;
}

}  // namespace

namespace sanatan {
ProfileEvents& profile_events() {
  static thread_local ProfileEvents ev;
  return ev;
}
}  // namespace sanatan

extern "C" {

const char* sanatan_status_string(int status) {
  switch (status) {
    case SANATAN_OK: return "ok";
    case SANATAN_ERR_INVALID: return "invalid argument (null or misaligned pointer, negative size, bad enum)";
    case SANATAN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case SANATAN_ERR_CUDA: return "CUDA runtime error";
    case SANATAN_ERR_ARCH: return "device is not sm_103 (GB300)";
    case SANATAN_ERR_TIMEOUT: return "device-side bounded wait timed out";
    default: return "unknown status";
  }
}

int sanatan_abi_version(void) { return kAbiVersion; }

size_t sanatan_state_bytes(int layers, int heads, int d, int dv) {
  if (layers < 0 || heads < 0 || d < 0 || dv < 0) return 0;
  return static_cast<size_t>(layers) * heads * (6ull * d * dv + 6ull * d) * sizeof(float);
}

int sanatan_featurize(const void* u, int u_dtype, const float* gamma, const float* omega,
                      const float* phi, int B, int H, int T, int d, int64_t pos0, void* out,
                      int out_dtype, void* stream) {
  if (!ok_dtype(u_dtype) || !ok_dtype(out_dtype)) return SANATAN_ERR_INVALID;
  if (B < 0 || H < 0 || T < 0 || d <= 0) return SANATAN_ERR_INVALID;
  if (d != 64) return SANATAN_ERR_UNSUPPORTED;
  const int64_t n = static_cast<int64_t>(B) * H * T;
  if (n == 0) return SANATAN_OK;
  if (!ok_ptr(u) || !ok_ptr(out)) return SANATAN_ERR_INVALID;
  if (int s = check_params(gamma, omega, phi)) return s;
  if (n * d / 256 + 1 > 0x7fffffffLL) return SANATAN_ERR_UNSUPPORTED;
  if (int s = check_arch()) return s;
  return from_cuda(featurize_launch(u, u_dtype, gamma, omega, phi, B, H, T, d, pos0, out,
                                    out_dtype, static_cast<cudaStream_t>(stream)));
}

int sanatan_rate_from_raw(const float* lambda_raw, int n, float scale, float* phi, void* stream) {
  if (n < 0) return SANATAN_ERR_INVALID;
  if (n == 0) return SANATAN_OK;
  if (!ok_ptr(lambda_raw) || !ok_ptr(phi)) return SANATAN_ERR_INVALID;
  if (int s = check_arch()) return s;
  return from_cuda(rate_launch(lambda_raw, nullptr, n, scale, phi,
                               static_cast<cudaStream_t>(stream)));
}

int sanatan_rate_from_raw_bwd(const float* lambda_raw, const float* dphi, int n, float scale,
                              float* dlambda_raw, void* stream) {
  if (n < 0) return SANATAN_ERR_INVALID;
  if (n == 0) return SANATAN_OK;
  if (!ok_ptr(lambda_raw) || !ok_ptr(dphi) || !ok_ptr(dlambda_raw)) return SANATAN_ERR_INVALID;
  if (int s = check_arch()) return s;
  return from_cuda(rate_launch(lambda_raw, dphi, n, scale, dlambda_raw,
                               static_cast<cudaStream_t>(stream)));
}

float sanatan_eps_raw(float eps, int d, int convention) {
  if (d <= 0) return -1.0f;
  if (convention == 0) return (4.0f * static_cast<float>(d) + 1e-6f) * eps;
  if (convention == 1) return (4.0f * static_cast<float>(d) * 1e-6f) * eps;
  return -1.0f;
}

size_t sanatan_chunk_fwd_workspace_size(int B, int H, int T, int d, int dv, int in_dtype) {
  if (B < 0 || H < 0 || T < 0 || d != 64 || dv != 64) return 0;
  if (in_dtype != SANATAN_BF16) return 0;
  return chunk_fwd_tc_workspace_bytes(B, H, T);
}

int sanatan_chunk_fwd_plan(int B, int H, int T, int in_dtype, int has_initial_state,
                           int* segments, int* launches) {
  if (!ok_dtype(in_dtype) || B < 0 || H < 0 || T < 0 || segments == nullptr || launches == nullptr)
    return SANATAN_ERR_INVALID;
  if (static_cast<int64_t>(B) * H == 0) {
    *segments = 0;
    *launches = 0;
    return SANATAN_OK;
  }
  if (in_dtype == SANATAN_F32) {
    *segments = 1;
    *launches = 1;
    return SANATAN_OK;
  }
  const int nseg = tc_segments(B, H, T);
  *segments = nseg;
  (void)has_initial_state;
  *launches = 1 + (nseg > 1 ? 1 : 0);
  return SANATAN_OK;
}

int sanatan_chunk_fwd(const void* q, const void* k, const void* v, int in_dtype,
                      const float* gamma, const float* omega, const float* phi, int B, int H,
                      int T, int d, int dv, int64_t pos0, float eps, const float* S0,
                      const float* z0, float* o, float* D, float* S_out, float* z_out,
                      void* workspace, size_t workspace_bytes, void* stream) {
  return sanatan::chunk_fwd_checked(q, k, v, in_dtype, gamma, omega, phi, B, H, T, d, dv, pos0,
                                    eps, S0, z0, o, D, S_out, z_out, workspace, workspace_bytes,
                                    stream, false);
}

}  // extern "C"

namespace sanatan {
// Argument checks and dispatch of sanatan_chunk_fwd.  With `fewer_segments`
// a workspace smaller than sanatan_chunk_fwd_workspace_size is accepted and
// the tensor-core path splits sequences into as many segments as it holds.
int chunk_fwd_checked(const void* q, const void* k, const void* v, int in_dtype,
                      const float* gamma, const float* omega, const float* phi, int B, int H,
                      int T, int d, int dv, int64_t pos0, float eps, const float* S0,
                      const float* z0, float* o, float* D, float* S_out, float* z_out,
                      void* workspace, size_t workspace_bytes, void* stream, bool fewer_segments) {
  if (!ok_dtype(in_dtype)) return SANATAN_ERR_INVALID;
  if (int s = check_sizes(B, H, T, d, dv)) return s;
  if ((S0 == nullptr) != (z0 == nullptr)) return SANATAN_ERR_INVALID;
  if ((S_out == nullptr) != (z_out == nullptr)) return SANATAN_ERR_INVALID;
  if (!ok_nullable(S0) || !ok_nullable(z0) || !ok_nullable(S_out) || !ok_nullable(z_out) ||
      !ok_nullable(D) || !ok_nullable(workspace))
    return SANATAN_ERR_INVALID;
  if (static_cast<int64_t>(B) * H == 0) return SANATAN_OK;
  if (T > 0 && (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(o))) return SANATAN_ERR_INVALID;
  if (int s = check_params(gamma, omega, phi)) return s;
  if (!fewer_segments &&
      workspace_bytes < sanatan_chunk_fwd_workspace_size(B, H, T, d, dv, in_dtype))
    return SANATAN_ERR_INVALID;
  if (int s = check_arch()) return s;
  ChunkFwdArgs a{q, k, v, in_dtype, gamma, omega, phi, B, H, T, d, dv, pos0, eps,
                 S0, z0, o, D, S_out, z_out, workspace, workspace_bytes};
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (in_dtype == SANATAN_BF16) return from_cuda(chunk_fwd_tc_launch(a, st));
  return from_cuda(chunk_fwd_simt_launch(a, st));
}
}  // namespace sanatan

extern "C" {

size_t sanatan_chunk_bwd_workspace_size(int B, int H, int T, int d, int dv, int in_dtype) {
  if (B < 0 || H < 0 || T < 0 || d != 64 || dv != 64) return 0;
  if (in_dtype != SANATAN_BF16) return 0;
  return chunk_bwd_tc_workspace_bytes(B, H, T);
}

int sanatan_chunk_bwd(const void* q, const void* k, const void* v, int in_dtype,
                      const float* gamma, const float* omega, const float* phi, int B, int H,
                      int T, int d, int dv, int64_t pos0, float eps, const float* S0,
                      const float* z0, const float* o, const float* D, const void* dO,
                      int grad_dtype, void* dq, void* dk, void* dv_out, float* dgamma,
                      float* domega, float* dphi, void* workspace, size_t workspace_bytes,
                      const void* fwd_workspace, size_t fwd_workspace_bytes, void* stream) {
  if (!ok_dtype(in_dtype) || !ok_dtype(grad_dtype)) return SANATAN_ERR_INVALID;
  if (!ok_nullable(fwd_workspace)) return SANATAN_ERR_INVALID;
  if (int s = check_sizes(B, H, T, d, dv)) return s;
  if ((S0 == nullptr) != (z0 == nullptr)) return SANATAN_ERR_INVALID;
  if (!ok_nullable(S0) || !ok_nullable(z0) || !ok_nullable(dphi) || !ok_nullable(workspace))
    return SANATAN_ERR_INVALID;
  if (H > 0 && (!ok_ptr(dgamma) || !ok_ptr(domega))) return SANATAN_ERR_INVALID;
  if (static_cast<int64_t>(B) * H * T > 0 &&
      (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(o) || !ok_ptr(D) || !ok_ptr(dO) ||
       !ok_ptr(dq) || !ok_ptr(dk) || !ok_ptr(dv_out)))
    return SANATAN_ERR_INVALID;
  if (H > 0) {
    if (int s = check_params(gamma, omega, phi)) return s;
  }
  if (workspace_bytes < sanatan_chunk_bwd_workspace_size(B, H, T, d, dv, in_dtype))
    return SANATAN_ERR_INVALID;
  if (H == 0) return SANATAN_OK;
  if (int s = check_arch()) return s;
  ChunkBwdArgs a{};
  a.f = ChunkFwdArgs{q, k, v, in_dtype, gamma, omega, phi, B, H, T, d, dv, pos0, eps,
                     S0, z0, nullptr, nullptr, nullptr, nullptr, workspace, workspace_bytes};
  a.o = o;
  a.Dn = D;
  a.dO = dO;
  a.grad_dtype = grad_dtype;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv_out;
  a.dgamma = dgamma;
  a.domega = domega;
  a.dphi = dphi;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.fwd_workspace = fwd_workspace;
  a.fwd_workspace_bytes = fwd_workspace == nullptr ? 0 : fwd_workspace_bytes;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (in_dtype == SANATAN_BF16) return from_cuda(chunk_bwd_tc_launch(a, st));
  return from_cuda(chunk_bwd_simt_launch(a, st));
}

size_t sanatan_power_fwd_workspace_size(int B, int H, int T, int d, int dv) {
  if (B < 0 || H < 0 || T < 0 || d != 64 || dv != 64) return 0;
  return pow_fwd_tc_workspace_bytes(B, H, T);
}

int sanatan_power_fwd(const void* q, const void* k, const void* v, const float* gamma,
                      const float* omega, const float* phi, int B, int H, int T, int d, int dv,
                      int64_t pos0, int p, float eps, float* o, float* D, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (int s = check_sizes(B, H, T, d, dv)) return s;
  if (p < 1) return SANATAN_ERR_INVALID;
  if (p > kMaxPower) return SANATAN_ERR_UNSUPPORTED;
  if (!ok_nullable(D)) return SANATAN_ERR_INVALID;
  if (static_cast<int64_t>(B) * H == 0 || T == 0) return SANATAN_OK;
  if (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(o) || !ok_ptr(workspace))
    return SANATAN_ERR_INVALID;
  if (int s = check_params(gamma, omega, phi)) return s;
  if (workspace_bytes < pow_fwd_tc_workspace_bytes(B, H, T)) return SANATAN_ERR_INVALID;
  if (static_cast<int64_t>(B) * H * ((T + 127) / 128) > 0x3fffffffLL) return SANATAN_ERR_UNSUPPORTED;
  if (int s = check_arch()) return s;
  PowFwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.gamma = gamma;
  a.omega = omega;
  a.phi = phi;
  a.B = B;
  a.H = H;
  a.T = T;
  a.pos0 = pos0;
  a.p = p;
  a.eps = eps;
  a.o = o;
  a.D = D;
  a.workspace = workspace;
  return from_cuda(pow_fwd_tc_launch(a, static_cast<cudaStream_t>(stream)));
}

int sanatan_ablation_fwd(const void* q, const void* k, const void* v, const float* gamma,
                         const float* omega, const float* phi, int B, int H, int T, int d,
                         int dv, int64_t pos0, int p, int channels, float shift, float eps,
                         float* o, float* D, void* workspace, size_t workspace_bytes,
                         void* stream) {
  if (int s = check_sizes(B, H, T, d, dv)) return s;
  if (channels != 3 && channels != 4) return SANATAN_ERR_INVALID;
  if (!(shift >= 0.0f) || (channels == 4 && shift != 0.0f)) return SANATAN_ERR_INVALID;
  if (p < 1) return SANATAN_ERR_INVALID;
  if (p != 1 && p != 2 && p != 4) return SANATAN_ERR_UNSUPPORTED;
  if (!ok_nullable(D)) return SANATAN_ERR_INVALID;
  if (static_cast<int64_t>(B) * H == 0 || T == 0) return SANATAN_OK;
  if (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(o) || !ok_ptr(workspace))
    return SANATAN_ERR_INVALID;
  if (int s = check_params(gamma, omega, phi)) return s;
  if (workspace_bytes < pow_fwd_tc_workspace_bytes(B, H, T)) return SANATAN_ERR_INVALID;
  if (static_cast<int64_t>(B) * H * ((T + 127) / 128) > 0x3fffffffLL) return SANATAN_ERR_UNSUPPORTED;
  if (int s = check_arch()) return s;
  PowFwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.gamma = gamma;
  a.omega = omega;
  a.phi = phi;
  a.B = B;
  a.H = H;
  a.T = T;
  a.pos0 = pos0;
  a.p = p;
  a.eps = eps;
  a.o = o;
  a.D = D;
  a.workspace = workspace;
  return from_cuda(ablation_fwd_tc_launch(a, channels, shift, static_cast<cudaStream_t>(stream)));
}

size_t sanatan_power_bwd_workspace_size(int B, int H, int T, int d, int dv) {
  if (B < 0 || H < 0 || T < 0 || d != 64 || dv != 64) return 0;
  return pow_bwd_tc_workspace_bytes(B, H, T);
}

int sanatan_power_bwd(const void* q, const void* k, const void* v, const float* gamma,
                      const float* omega, const float* phi, int B, int H, int T, int d, int dv,
                      int64_t pos0, int p, float eps, const float* o, const float* D,
                      const void* dO, int grad_dtype, void* dq, void* dk, void* dv_out,
                      float* dgamma, float* domega, float* dphi, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (int s = check_sizes(B, H, T, d, dv)) return s;
  if (p < 1 || !ok_dtype(grad_dtype)) return SANATAN_ERR_INVALID;
  if (p > kMaxPower) return SANATAN_ERR_UNSUPPORTED;
  if (H > 0 && (!ok_ptr(dgamma) || !ok_ptr(domega) || !ok_nullable(dphi)))
    return SANATAN_ERR_INVALID;
  if (H > 0) {
    if (int s = check_params(gamma, omega, phi)) return s;
  }
  if (static_cast<int64_t>(B) * H > 0 && T > 0) {
    if (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(o) || !ok_ptr(D) || !ok_ptr(dO) ||
        !ok_ptr(dq) || !ok_ptr(dk) || !ok_ptr(dv_out) || !ok_ptr(workspace))
      return SANATAN_ERR_INVALID;
    if (workspace_bytes < pow_bwd_tc_workspace_bytes(B, H, T)) return SANATAN_ERR_INVALID;
    if (static_cast<int64_t>(B) * H * ((T + 127) / 128) > 0x3fffffffLL)
      return SANATAN_ERR_UNSUPPORTED;
  }
  if (H == 0) return SANATAN_OK;
  if (int s = check_arch()) return s;
  PowBwdArgs a;
  a.f.q = q;
  a.f.k = k;
  a.f.v = v;
  a.f.gamma = gamma;
  a.f.omega = omega;
  a.f.phi = phi;
  a.f.B = B;
  a.f.H = H;
  a.f.T = T;
  a.f.pos0 = pos0;
  a.f.p = p;
  a.f.eps = eps;
  a.f.workspace = workspace;
  a.o = o;
  a.D = D;
  a.dO = dO;
  a.grad_dtype = grad_dtype;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv_out;
  a.dgamma = dgamma;
  a.domega = domega;
  a.dphi = dphi;
  return from_cuda(pow_bwd_tc_launch(a, static_cast<cudaStream_t>(stream)));
}

int sanatan_set_profile_events(void* start, void* stop) {
  if ((start == nullptr) != (stop == nullptr)) return SANATAN_ERR_INVALID;
  profile_events().start = static_cast<cudaEvent_t>(start);
  profile_events().stop = static_cast<cudaEvent_t>(stop);
  return SANATAN_OK;
}

int sanatan_device_status(void* stream) {
  if (int s = check_arch()) return s;
  const int h = tc_read_and_clear_error(static_cast<cudaStream_t>(stream));
  const int hb = bwd_tc_read_and_clear_error(static_cast<cudaStream_t>(stream));
  const int hp = pow_tc_read_and_clear_error(static_cast<cudaStream_t>(stream));
  const int hpb = pow_bwd_tc_read_and_clear_error(static_cast<cudaStream_t>(stream));
  const int hs = stack_read_and_clear_error(static_cast<cudaStream_t>(stream));
  if (h < 0 || hb < 0 || hp < 0 || hpb < 0 || hs < 0) return SANATAN_ERR_CUDA;
  if (hb || hp || hpb || hs) return SANATAN_ERR_TIMEOUT;
  return h ? SANATAN_ERR_TIMEOUT : SANATAN_OK;
}

size_t sanatan_state_bytes_harmonic(int layers, int heads, int d, int dv, int harmonics) {
  if (layers < 0 || heads < 0 || d < 0 || dv < 0 || harmonics < 1) return 0;
  const size_t F = static_cast<size_t>(2 * (2 * harmonics + 1)) * d;
  return static_cast<size_t>(layers) * heads * (F * dv + F) * sizeof(float);
}

int sanatan_featurize_harmonic(const void* u, int u_dtype, const float* gamma, const float* omega,
                               const float* phi, int B, int H, int T, int d, int64_t pos0,
                               int harmonics, void* out, int out_dtype, void* stream) {
  if (!ok_dtype(u_dtype) || !ok_dtype(out_dtype)) return SANATAN_ERR_INVALID;
  if (B < 0 || H < 0 || T < 0 || d <= 0 || harmonics < 1) return SANATAN_ERR_INVALID;
  if (d != 64 || harmonics > 3) return SANATAN_ERR_UNSUPPORTED;
  const int64_t n = static_cast<int64_t>(B) * H * T;
  if (n == 0) return SANATAN_OK;
  if (!ok_ptr(u) || !ok_ptr(out)) return SANATAN_ERR_INVALID;
  if (int s = check_params(gamma, omega, phi)) return s;
  if (n * d / 256 + 1 > 0x7fffffffLL) return SANATAN_ERR_UNSUPPORTED;
  if (int s = check_arch()) return s;
  HarmonicFeatArgs a{u, u_dtype, gamma, omega, phi, B, H, T, pos0, harmonics, out, out_dtype};
  return from_cuda(featurize_harmonic_launch(a, static_cast<cudaStream_t>(stream)));
}

int sanatan_chunk_fwd_harmonic(const void* q, const void* k, const void* v, int in_dtype,
                               const float* gamma, const float* omega, const float* phi, int B,
                               int H, int T, int d, int dv, int64_t pos0, int harmonics,
                               float eps, const float* S0, const float* z0, float* o, float* D,
                               float* S_out, float* z_out, void* stream) {
  if (!ok_dtype(in_dtype) || harmonics < 1) return SANATAN_ERR_INVALID;
  if (int s = check_sizes(B, H, T, d, dv)) return s;
  if (harmonics > 3) return SANATAN_ERR_UNSUPPORTED;
  if ((S0 == nullptr) != (z0 == nullptr)) return SANATAN_ERR_INVALID;
  if ((S_out == nullptr) != (z_out == nullptr)) return SANATAN_ERR_INVALID;
  if (!ok_nullable(S0) || !ok_nullable(z0) || !ok_nullable(S_out) || !ok_nullable(z_out) ||
      !ok_nullable(D))
    return SANATAN_ERR_INVALID;
  if (static_cast<int64_t>(B) * H == 0) return SANATAN_OK;
  if (T > 0 && (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(o))) return SANATAN_ERR_INVALID;
  if (int s = check_params(gamma, omega, phi)) return s;
  if (int s = check_arch()) return s;
  ChunkFwdArgs a{q, k, v, in_dtype, gamma, omega, phi, B, H, T, d, dv, pos0, eps,
                 S0, z0, o, D, S_out, z_out, nullptr, 0};
  return from_cuda(chunk_fwd_harmonic_launch(a, harmonics, static_cast<cudaStream_t>(stream)));
}

size_t sanatan_chunk_bwd_harmonic_workspace_size(int B, int H, int T, int d, int dv,
                                                 int harmonics) {
  if (B < 0 || H < 0 || T < 0 || d != 64 || dv != 64 || harmonics < 1 || harmonics > 3) return 0;
  return chunk_bwd_harmonic_workspace_bytes(B, H, T, harmonics);
}

int sanatan_chunk_bwd_harmonic(const void* q, const void* k, const void* v, int in_dtype,
                               const float* gamma, const float* omega, const float* phi, int B,
                               int H, int T, int d, int dv, int64_t pos0, int harmonics,
                               float eps, const float* S0, const float* z0, const float* o,
                               const float* D, const void* dO, int grad_dtype, void* dq, void* dk,
                               void* dv_out, float* dgamma, float* domega, float* dphi,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (!ok_dtype(in_dtype) || !ok_dtype(grad_dtype) || harmonics < 1) return SANATAN_ERR_INVALID;
  if (int s = check_sizes(B, H, T, d, dv)) return s;
  if (harmonics > 3) return SANATAN_ERR_UNSUPPORTED;
  if ((S0 == nullptr) != (z0 == nullptr)) return SANATAN_ERR_INVALID;
  if (!ok_nullable(S0) || !ok_nullable(z0) || !ok_nullable(dphi) || !ok_nullable(workspace))
    return SANATAN_ERR_INVALID;
  if (H > 0 && (!ok_ptr(dgamma) || !ok_ptr(domega))) return SANATAN_ERR_INVALID;
  if (static_cast<int64_t>(B) * H * T > 0 &&
      (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(o) || !ok_ptr(D) || !ok_ptr(dO) ||
       !ok_ptr(dq) || !ok_ptr(dk) || !ok_ptr(dv_out)))
    return SANATAN_ERR_INVALID;
  if (H > 0) {
    if (int s = check_params(gamma, omega, phi)) return s;
  }
  const size_t need = sanatan_chunk_bwd_harmonic_workspace_size(B, H, T, d, dv, harmonics);
  if (workspace_bytes < need || (need > 0 && workspace == nullptr)) return SANATAN_ERR_INVALID;
  if (H == 0) return SANATAN_OK;
  if (int s = check_arch()) return s;
  ChunkBwdArgs a{};
  a.f = ChunkFwdArgs{q, k, v, in_dtype, gamma, omega, phi, B, H, T, d, dv, pos0, eps,
                     S0, z0, nullptr, nullptr, nullptr, nullptr, nullptr, 0};
  a.o = o;
  a.Dn = D;
  a.dO = dO;
  a.grad_dtype = grad_dtype;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv_out;
  a.dgamma = dgamma;
  a.domega = domega;
  a.dphi = dphi;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  return from_cuda(
      chunk_bwd_harmonic_launch(a, harmonics, static_cast<cudaStream_t>(stream)));
}

int sanatan_decode_step_harmonic(float* S, float* z, const float* q, const float* k,
                                 const float* v, const float* gamma, const float* omega,
                                 const float* phi, const int64_t* pos, int N, int G, int d, int dv,
                                 int harmonics, float eps, float* o, void* stream) {
  if (N < 0 || G <= 0 || d < 0 || dv < 0 || harmonics < 1) return SANATAN_ERR_INVALID;
  if (d != 64 || dv != 64 || harmonics > 3) return SANATAN_ERR_UNSUPPORTED;
  if (N == 0) return SANATAN_OK;
  if (!ok_ptr(S) || !ok_ptr(z) || !ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(pos) ||
      !ok_ptr(o))
    return SANATAN_ERR_INVALID;
  if (int s = check_params(gamma, omega, phi)) return s;
  if (static_cast<int64_t>(N) * 4 > 0x7fffffffLL) return SANATAN_ERR_UNSUPPORTED;
  if (int s = check_arch()) return s;
  return from_cuda(decode_harmonic_launch(S, z, q, k, v, gamma, omega, phi, pos, N, G, eps,
                                          harmonics, o, static_cast<cudaStream_t>(stream)));
}

size_t sanatan_stack_decode_workspace_size(int B, int heads, int d) {
  if (B < 0 || heads < 0 || d != 64) return 0;
  return stack_workspace_bytes(B, heads, d);
}

int sanatan_stack_decode_step(float* x, const float* Wqkv, const float* Wo, float* S, float* z,
                              const float* gamma, const float* omega, const float* phi,
                              const int64_t* pos, int B, int L, int heads, int d, float eps,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || L < 0 || heads < 0 || d < 0) return SANATAN_ERR_INVALID;
  if (d != 64 || B > stack_max_batch() || (heads * d) % 128 != 0) return SANATAN_ERR_UNSUPPORTED;
  if (B == 0 || L == 0 || heads == 0) return SANATAN_OK;
  if (!ok_ptr(x) || !ok_ptr(Wqkv) || !ok_ptr(Wo) || !ok_ptr(S) || !ok_ptr(z) || !ok_ptr(pos) ||
      !ok_ptr(workspace))
    return SANATAN_ERR_INVALID;
  if (int s = check_params(gamma, omega, phi)) return s;
  if (workspace_bytes < stack_workspace_bytes(B, heads, d)) return SANATAN_ERR_INVALID;
  if (int s = check_arch()) return s;
  StackArgs a{x, Wqkv, Wo, S, z, gamma, omega, phi, pos, B, L, heads, eps, workspace};
  return from_cuda(stack_decode_launch(a, static_cast<cudaStream_t>(stream)));
}

int sanatan_selftest_wait_timeout(uint64_t timeout_ns, int arrive, void* stream) {
  if (timeout_ns < 1000ull || timeout_ns > 1000000000ull) return SANATAN_ERR_INVALID;
  if (arrive != 0 && arrive != 1) return SANATAN_ERR_INVALID;
  if (int s = check_arch()) return s;
  return from_cuda(tc_timeout_probe_launch(timeout_ns, arrive, static_cast<cudaStream_t>(stream)));
}

int sanatan_decode_step(float* S, float* z, const float* q, const float* k, const float* v,
                        const float* gamma, const float* omega, const float* phi,
                        const int64_t* pos, int N, int G, int d, int dv, float eps, float* o,
                        void* stream) {
  if (N < 0 || G <= 0 || d < 0 || dv < 0) return SANATAN_ERR_INVALID;
  if (d != 64 || dv != 64) return SANATAN_ERR_UNSUPPORTED;
  if (N == 0) return SANATAN_OK;
  if (!ok_ptr(S) || !ok_ptr(z) || !ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(pos) ||
      !ok_ptr(o))
    return SANATAN_ERR_INVALID;
  if (int s = check_params(gamma, omega, phi)) return s;
  if (int s = check_arch()) return s;
  return from_cuda(decode_step_launch(S, z, q, k, v, gamma, omega, phi, pos, N, G, eps, o,
                                      static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
