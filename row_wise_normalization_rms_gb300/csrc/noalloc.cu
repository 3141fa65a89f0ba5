// rms_bwd_noalloc: the backward with its column-partial workspace in a
// fixed device array owned by this library instead of a caller buffer.
//
// For callers that cannot obtain device memory for scratch themselves: a
// plugin inside a host program whose allocator owns all device memory and
// offers plugins no scratch requests, or a latency-critical loop that must
// not pay cudaMalloc's device-wide synchronisation.  Inputs and outputs are
// still the caller's.
//
// The array below is allocated when this library's module is loaded on a
// device and is held by every device that loads the library until the
// process exits.  Host code may not pass the array's name to a kernel (on
// the host it is only a stand-in symbol), so the first call on each device
// looks up its device address with cudaGetSymbolAddress, with that device
// current, and caches it; that first call should therefore happen before
// any stream capture.  A device reset (cudaDeviceReset) unloads the module
// and leaves the cached address stale: do not call this entry point on a
// device after resetting it in the same process.  All calls on a device share the one array: calls
// whose executions overlap on the GPU (different streams, or concurrent
// host threads) race on it and must be serialised by the caller.  Nothing
// in it needs clearing between calls: every partial row the column
// reduction reads is fully written earlier in the same call.
#include <mutex>

#include "rmsnorm.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[RMS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up
// once per device).
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" rms_status rms_bwd_noalloc(void* dy, const void* x, const void* gamma,
                                      const float* rstd, void* dx, float* dgamma, int64_t M,
                                      int64_t N, rms_dtype dtype, int gemma, int inplace_dx,
                                      void* stream) {
  // No rows (or a bad shape): rms_bwd answers without a workspace (M == 0
  // zeroes dgamma), so the scratch array is not looked up at all.
  if (M <= 0 || N <= 0)
    return rms_bwd_ex(dy, x, gamma, rstd, dx, dgamma, nullptr, 0, M, N, dtype, gemma, inplace_dx,
                      RMS_PATH_AUTO, stream);
  const size_t need = rms_bwd_workspace_size(M, N);
  if (need == 0) return RMS_ERR_CUDA;  // the current device could not be queried
  if (need > (size_t)RMS_NOALLOC_SCRATCH_BYTES) return RMS_ERR_WORKSPACE;
  void* ws = scratch_on_current_device();
  if (!ws) return RMS_ERR_CUDA;
  return rms_bwd_ex(dy, x, gamma, rstd, dx, dgamma, ws, (size_t)RMS_NOALLOC_SCRATCH_BYTES, M, N,
                    dtype, gemma, inplace_dx, RMS_PATH_AUTO, stream);
}
