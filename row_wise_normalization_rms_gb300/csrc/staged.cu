// Staged mapping (rows staged in shared memory by cp.async.bulk) and the
// device status word its bounded waits report through.
#include "common.cuh"
#include "internal.h"

namespace rmsk {

// Nonzero once a bounded wait gave up; read and cleared by the host.
__device__ int g_rms_device_status = 0;

}  // namespace rmsk

namespace rmsi {

bool plan_staged(int N, int dtype, bool bwd, const DeviceInfo& d, Mapping* m) {
  (void)N; (void)dtype; (void)bwd; (void)d; (void)m;
  return false;
}

cudaError_t launch_fwd_staged(const FwdArgs&, const Mapping&, const DeviceInfo&, long long,
                              cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t size_bwd_staged(const BwdArgs&, const DeviceInfo&, Mapping*) {
  return cudaErrorNotSupported;
}

cudaError_t launch_bwd_staged(const BwdArgs&, const Mapping&, const DeviceInfo&, long long,
                              cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t take_device_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, rmsk::g_rms_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(rmsk::g_rms_device_status, &zero, sizeof(int));
    if (e != cudaSuccess) return e;
  }
  *status = v;
  return cudaSuccess;
}

}  // namespace rmsi
