// sanatan_chunk_fwd_noalloc: the tensor-core chunked forward with its scratch
// in a fixed, library-owned device array instead of a caller-provided
// workspace, for callers that cannot allocate device memory themselves.
#include <mutex>

#include "sanatan_internal.h"

namespace sanatan {
namespace {

// The scratch of the segment split (per-segment state sums of every segment
// but the last, 321 x 80 floats per (sequence, segment)).  16 MiB holds 163
// such slots.  A problem whose preferred split needs more is run with as many
// segments as the array holds; one segment needs no scratch at all, so every
// problem size runs.  Every GPU that loads the library keeps this array until
// the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// The array's name is a host-side stand-in in host code: the kernels must be
// given the device address, looked up once per device with that device
// current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace sanatan

extern "C" size_t sanatan_chunk_fwd_noalloc_max_scratch_bytes(void) {
  return sanatan::kNoAllocScratchBytes;
}

extern "C" int sanatan_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                         const float* gamma, const float* omega,
                                         const float* phi, int B, int H, int T, int d, int dv,
                                         int64_t pos0, float eps, const float* S0,
                                         const float* z0, float* o, float* D, float* S_out,
                                         float* z_out, void* stream) {
  using namespace sanatan;
  if (B < 0 || H < 0 || T < 0 || d < 0 || dv < 0) return SANATAN_ERR_INVALID;
  if (d != 64 || dv != 64) return SANATAN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * H > (1LL << 31) - 1) return SANATAN_ERR_UNSUPPORTED;
  // The split is chosen to fit the array (tc_segments_fit); the check below
  // only guards that contract.
  const int nseg = tc_segments_fit(B, H, T, kNoAllocScratchBytes);
  const size_t need = nseg > 1 ? static_cast<size_t>(B) * H * nseg * 321 * 80 * sizeof(float) : 0;
  if (need > kNoAllocScratchBytes) return SANATAN_ERR_UNSUPPORTED;  // beyond the fixed scratch
  void* scratch = nullptr;
  if (need > 0) {
    if (scratch_address(&scratch) != cudaSuccess) return SANATAN_ERR_CUDA;
    if (!aligned16(scratch)) return SANATAN_ERR_CUDA;
  }
  // Argument checks, dispatch and launches are those of sanatan_chunk_fwd.
  return chunk_fwd_checked(q, k, v, SANATAN_BF16, gamma, omega, phi, B, H, T, d, dv, pos0, eps,
                           S0, z0, o, D, S_out, z_out, scratch, kNoAllocScratchBytes, stream, true);
}
