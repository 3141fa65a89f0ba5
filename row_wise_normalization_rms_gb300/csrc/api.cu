// C ABI of librmsnorm.so: argument validation, row-mapping dispatch,
// workspace sizing and status reporting.  Nothing here allocates device
// memory or touches tensor data; every error is found before a launch.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "internal.h"
#include "rmsnorm.h"

namespace {

using rmsi::BwdArgs;
using rmsi::DeviceInfo;
using rmsi::FwdArgs;
using rmsi::Mapping;

constexpr long long kDefaultWaitLimit = 1ll << 22;
std::atomic<long long> g_wait_limit{kDefaultWaitLimit};
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ok[kMaxDevices] = {};

bool current_device(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev_ok[dev]) {
    DeviceInfo d;
    d.device = dev;
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    d.sms = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return false;
    d.smem_optin = (size_t)v;
    g_dev[dev] = d;
    g_dev_ok[dev] = true;
  }
  *out = g_dev[dev];
  return true;
}

// (kernel, device) pairs whose dynamic shared memory limit is already raised.
std::mutex g_optin_mu;
std::set<std::pair<const void*, int>> g_optin;

int elem_bytes(int dtype) { return rmsi::dtype_bytes(dtype); }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Half-open byte ranges [p, p + n) overlap.
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

bool valid_common(int64_t M, int64_t N, rms_dtype dtype, int gemma) {
  if (dtype < RMS_F32 || dtype > RMS_F16_W32) return false;
  if (gemma != 0 && gemma != 1) return false;
  if (M < 0 || N <= 0) return false;
  return true;
}

// Matrix byte count, or 0 when M*N*b does not fit in an int64.
size_t matrix_bytes(int64_t M, int64_t N, int b) {
  if (M == 0) return 0;
  if (N > INT64_MAX / b || M > INT64_MAX / (N * b)) return 0;
  return (size_t)(M * N * b);
}

size_t workspace_need(int64_t M, int64_t N, const DeviceInfo& d) {
  int64_t P = rmsi::max_partials(d.sms);
  if (P > M) P = M;
  const size_t bytes = (size_t)P * (size_t)N * sizeof(float);
  return (bytes + 255) / 256 * 256;
}

// Row bytes above which the automatic choice stages rows in shared memory
// instead of holding them in registers, from GB300 timings over N = 512 ..
// 16384 bf16: the forward (one stream in, one out) is fastest in registers
// up to 16 KiB rows; the backward (two streams in) gains from the deeper
// copy pipeline as soon as rows exceed 1 KiB.
constexpr int64_t kAutoStagedRowBytesFwd = 16384;
constexpr int64_t kAutoStagedRowBytesBwd = 1024;
constexpr int kAutoChunkedClusterFwd = 2;
constexpr int64_t kAutoChunkedRowBytesBwd = 65536;

bool prefer_staged(int N, int dtype, bool bwd) {
  const int64_t row = (int64_t)N * elem_bytes(dtype);
  return row > (bwd ? kAutoStagedRowBytesBwd : kAutoStagedRowBytesFwd);
}

// Picks the row mapping for a call.  A forced path that cannot take the
// shape is an error, never a silent switch.
// With a fused residual the register forward holds twice the vectors and is
// built for at most 512 threads per CTA.
bool plan_registers_for(int N, int dtype, bool bwd, bool res, Mapping* m) {
  return rmsi::plan_registers(N, dtype, bwd, m) && !(res && !bwd && m->threads > 512);
}

rms_status choose(rms_path path, int N, int dtype, bool bwd, bool aligned, const DeviceInfo& d,
                  Mapping* m, bool res = false, int64_t M = 0) {
  switch (path) {
    case RMS_PATH_AUTO:
      if (aligned && prefer_staged(N, dtype, bwd) && rmsi::plan_staged(N, dtype, bwd, d, m, res, M)) {
        // A row the staged mapping splits over a cluster waits on a cluster
        // barrier per row; the chunked mapping's one-pass cluster kernels
        // overlap that exchange with the next row's loads.  They take
        // forward rows the staged mapping splits at all and backward rows of
        // 64 KiB and more (GB300 bf16: N = 65536 fwd 86 % of HBM against
        // 68 %, N = 32768 bwd 86 % against 62 %; the 2-CTA staged backward
        // at N = 11008 .. 16384 runs at 85-96 % against 75-86 %).
        const bool wide = bwd ? (m->cluster > 1 && (int64_t)N * elem_bytes(dtype) >=
                                                       kAutoChunkedRowBytesBwd)
                              : m->cluster >= kAutoChunkedClusterFwd;
        if (wide && rmsi::plan_chunked(N, dtype, bwd, res, m)) return RMS_OK;
        return RMS_OK;
      }
      if (aligned && plan_registers_for(N, dtype, bwd, res, m)) return RMS_OK;
      if (aligned && rmsi::plan_staged(N, dtype, bwd, d, m, res, M)) return RMS_OK;
      if (aligned && rmsi::plan_chunked(N, dtype, bwd, res, m)) return RMS_OK;
      if (rmsi::plan_scalar(N, dtype, bwd, d, m)) return RMS_OK;
      return RMS_ERR_UNSUPPORTED;
    case RMS_PATH_REGISTERS:
      if (!aligned) return RMS_ERR_ALIGNMENT;
      return plan_registers_for(N, dtype, bwd, res, m) ? RMS_OK : RMS_ERR_UNSUPPORTED;
    case RMS_PATH_STAGED:
      if (!aligned) return RMS_ERR_ALIGNMENT;
      return rmsi::plan_staged(N, dtype, bwd, d, m, res, M) ? RMS_OK : RMS_ERR_UNSUPPORTED;
    case RMS_PATH_SCALAR:
      return rmsi::plan_scalar(N, dtype, bwd, d, m) ? RMS_OK : RMS_ERR_UNSUPPORTED;
    case RMS_PATH_CHUNKED:
      if (!aligned) return RMS_ERR_ALIGNMENT;
      return rmsi::plan_chunked(N, dtype, bwd, res, m) ? RMS_OK : RMS_ERR_UNSUPPORTED;
    default:
      return RMS_ERR_INVALID_ARG;
  }
}

// The backward's mapping for a call, with its grid and partial rows sized
// (m->partials workspace rows; *kbuf: where the three-pass chunked mapping
// keeps its per-row values).  Launches nothing; a.ws and a.dgamma are only
// used as addresses.
rms_status plan_bwd(const BwdArgs& a, rms_path path, bool aligned, const DeviceInfo& d,
                    Mapping* m, float** kbuf) {
  const rms_status st = choose(path, a.N, a.dtype, true, aligned, d, m, a.dh != nullptr, a.M);
  if (st != RMS_OK) return st;
  cudaError_t e = cudaSuccess;
  switch (m->path) {
    case rmsi::kRegisters: e = rmsi::size_bwd_registers(a, d, m); break;
    case rmsi::kStaged: e = rmsi::size_bwd_staged(a, d, m); break;
    case rmsi::kChunked:
      if (!rmsi::size_bwd_chunked(a, d, m, kbuf)) return RMS_ERR_UNSUPPORTED;
      break;
    default: e = rmsi::size_bwd_scalar(a, d, m); break;
  }
  return e == cudaSuccess ? RMS_OK : RMS_ERR_CUDA;
}

// Most rows whose terms one partial row sums: every mapping deals tiles of
// m.rows_per_cta consecutive rows to its m.partials work units in turn.
int64_t most_rows_per_partial(int64_t M, const Mapping& m) {
  const int64_t R = m.rows_per_cta > 0 ? m.rows_per_cta : 1;
  const int64_t tiles = (M + R - 1) / R;
  return R * ((tiles + m.partials - 1) / m.partials);
}

}  // namespace

namespace rmsi {

cudaError_t opt_in_max_smem(const void* kernel, const DeviceInfo& d) {
  std::lock_guard<std::mutex> lk(g_optin_mu);
  if (g_optin.count({kernel, d.device})) return cudaSuccess;
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  // Static plus dynamic shared memory may not exceed the opt-in maximum.
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(d.smem_optin - fa.sharedSizeBytes));
  if (e != cudaSuccess) return e;
  g_optin.insert({kernel, d.device});
  return cudaSuccess;
}

}  // namespace rmsi

extern "C" {

const char* rms_status_string(rms_status s) {
  switch (s) {
    case RMS_OK: return "ok";
    case RMS_ERR_INVALID_ARG: return "invalid argument";
    case RMS_ERR_UNSUPPORTED: return "unsupported shape for the requested row mapping";
    case RMS_ERR_ALIGNMENT: return "requested row mapping needs 16-byte aligned rows and pointers";
    case RMS_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case RMS_ERR_CUDA: return "CUDA runtime error";
    case RMS_ERR_TIMEOUT: return "device-side bounded wait gave up";
    default: return "unknown status";
  }
}

int64_t rms_set_wait_limit(int64_t polls) {
  const long long v = polls < 0 ? kDefaultWaitLimit : (long long)polls;
  return (int64_t)g_wait_limit.exchange(v);
}

uint64_t rms_launch_count(void) { return g_launches.load(); }

size_t rms_bwd_workspace_size(int64_t M, int64_t N) {
  if (M <= 0 || N <= 0) return 0;
  DeviceInfo d;
  if (!current_device(&d)) return 0;
  return workspace_need(M, N, d);
}

// The forward, with or without a fused residual add (res and h both given,
// or both NULL).
static rms_status fwd_impl(const void* x, const void* res, const void* gamma, void* y, void* h,
                           float* rstd, int64_t M, int64_t N, float eps, rms_dtype dtype, int gemma,
                    rms_path path, void* stream) {
  if (!valid_common(M, N, dtype, gemma)) return RMS_ERR_INVALID_ARG;
  if (!isfinite(eps) || eps < 0.f) return RMS_ERR_INVALID_ARG;
  if (path < RMS_PATH_AUTO || path > RMS_PATH_CHUNKED) return RMS_ERR_INVALID_ARG;
  if (N > (int64_t)INT32_MAX) return RMS_ERR_UNSUPPORTED;
  if (M == 0) return RMS_OK;
  if (!x || !gamma || !y || !rstd) return RMS_ERR_INVALID_ARG;
  const bool fused = res != nullptr || h != nullptr;
  if (fused && (!res || !h)) return RMS_ERR_INVALID_ARG;
  const int b = elem_bytes(dtype);
  const size_t xb = matrix_bytes(M, N, b);
  if (xb == 0) return RMS_ERR_INVALID_ARG;
  const size_t gb = (size_t)N * rmsi::weight_bytes(dtype), rb = (size_t)M * sizeof(float);
  // Written: y, rstd and (fused) h; h == res is the one sanctioned alias.
  const void* reads[3] = {x, gamma, res};
  const size_t read_n[3] = {xb, gb, xb};
  const void* writes[3] = {y, rstd, h};
  const size_t write_n[3] = {xb, rb, xb};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 3; ++j) {
      if (i == 2 && j == 2 && h == res) continue;
      if (overlap(writes[i], write_n[i], reads[j], read_n[j])) return RMS_ERR_INVALID_ARG;
    }
    for (int j = i + 1; j < 3; ++j)
      if (overlap(writes[i], write_n[i], writes[j], write_n[j])) return RMS_ERR_INVALID_ARG;
  }

  DeviceInfo d;
  if (!current_device(&d)) return RMS_ERR_CUDA;
  const bool aligned = (N * b) % 16 == 0 && aligned16(x) && aligned16(gamma) && aligned16(y) &&
                       (!fused || (aligned16(res) && aligned16(h)));
  Mapping m;
  const rms_status st = choose(path, (int)N, dtype, false, aligned, d, &m, fused, M);
  if (st != RMS_OK) return st;

  FwdArgs a{x, gamma, y, rstd, M, (int)N, eps, (int)dtype, gemma, res, h};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (m.path) {
    case rmsi::kRegisters:
      if ((M + m.rows_per_cta - 1) / m.rows_per_cta > INT32_MAX) return RMS_ERR_UNSUPPORTED;
      e = rmsi::launch_fwd_registers(a, m, s);
      break;
    case rmsi::kStaged:
      e = rmsi::launch_fwd_staged(a, m, d, g_wait_limit.load(), s);
      break;
    case rmsi::kChunked:
      e = rmsi::launch_fwd_chunked(a, m, d, g_wait_limit.load(), s);
      if (e == cudaSuccess && !m.wide) g_launches.fetch_add(1);  // three-pass: two kernels
      break;
    default:
      if (M > INT32_MAX) return RMS_ERR_UNSUPPORTED;
      e = rmsi::launch_fwd_scalar(a, m, s);
      break;
  }
  if (e != cudaSuccess) return RMS_ERR_CUDA;
  g_launches.fetch_add(1);
  return RMS_OK;
}

rms_status rms_fwd_ex(const void* x, const void* gamma, void* y, float* rstd, int64_t M,
                      int64_t N, float eps, rms_dtype dtype, int gemma, rms_path path,
                      void* stream) {
  return fwd_impl(x, nullptr, gamma, y, nullptr, rstd, M, N, eps, dtype, gemma, path, stream);
}

rms_status rms_fwd(const void* x, const void* gamma, void* y, float* rstd, int64_t M, int64_t N,
                   float eps, rms_dtype dtype, int gemma, void* stream) {
  return fwd_impl(x, nullptr, gamma, y, nullptr, rstd, M, N, eps, dtype, gemma, RMS_PATH_AUTO,
                  stream);
}

rms_status rms_fwd_add_ex(const void* x, const void* residual, const void* gamma, void* y,
                          void* h, float* rstd, int64_t M, int64_t N, float eps, rms_dtype dtype,
                          int gemma, rms_path path, void* stream) {
  if (M > 0 && (!residual || !h)) return RMS_ERR_INVALID_ARG;
  return fwd_impl(x, residual, gamma, y, h, rstd, M, N, eps, dtype, gemma, path, stream);
}

rms_status rms_fwd_add(const void* x, const void* residual, const void* gamma, void* y, void* h,
                       float* rstd, int64_t M, int64_t N, float eps, rms_dtype dtype, int gemma,
                       void* stream) {
  return rms_fwd_add_ex(x, residual, gamma, y, h, rstd, M, N, eps, dtype, gemma, RMS_PATH_AUTO,
                        stream);
}

// The backward, with or without a fused residual gradient dh (NULL: none).
static rms_status bwd_impl(void* dy, const void* x, const void* gamma, const float* rstd,
                           const void* dh, void* dx, float* dgamma, void* workspace,
                           size_t workspace_bytes, int64_t M, int64_t N, rms_dtype dtype,
                           int gemma, int inplace_dx, rms_path path, void* stream) {
  if (!valid_common(M, N, dtype, gemma)) return RMS_ERR_INVALID_ARG;
  if (inplace_dx != 0 && inplace_dx != 1) return RMS_ERR_INVALID_ARG;
  if (path < RMS_PATH_AUTO || path > RMS_PATH_CHUNKED) return RMS_ERR_INVALID_ARG;
  if (N > (int64_t)INT32_MAX) return RMS_ERR_UNSUPPORTED;
  if (inplace_dx) {
    if (dx && dx != dy) return RMS_ERR_INVALID_ARG;
    dx = dy;
  }
  if (!dgamma) return RMS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 0) {
    // The sum over zero rows: dgamma = 0.
    return cudaMemsetAsync(dgamma, 0, (size_t)N * sizeof(float), s) == cudaSuccess ? RMS_OK
                                                                                    : RMS_ERR_CUDA;
  }
  if (!dx || !dy || !x || !gamma || !rstd) return RMS_ERR_INVALID_ARG;
  const int b = elem_bytes(dtype);
  const size_t xb = matrix_bytes(M, N, b);
  if (xb == 0) return RMS_ERR_INVALID_ARG;
  const size_t gb = (size_t)N * rmsi::weight_bytes(dtype), rb = (size_t)M * sizeof(float),
               db = (size_t)N * sizeof(float);

  if (!workspace) return RMS_ERR_WORKSPACE;
  DeviceInfo d;
  if (!current_device(&d)) return RMS_ERR_CUDA;
  const size_t need = workspace_need(M, N, d);
  if (workspace_bytes < need || ((uintptr_t)workspace & 255u) != 0) return RMS_ERR_WORKSPACE;

  // Written ranges (dx, dgamma, workspace) must not overlap anything else;
  // dx == dy (inplace_dx) and dx == dh are the sanctioned aliases.
  const void* reads[5] = {x, gamma, rstd, dy, dh};
  const size_t read_n[5] = {xb, gb, rb, xb, xb};
  const void* writes[3] = {dx, dgamma, workspace};
  const size_t write_n[3] = {xb, db, need};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 5; ++j) {
      if (i == 0 && reads[j] == dx && (j == 3 || j == 4)) continue;
      if (overlap(writes[i], write_n[i], reads[j], read_n[j])) return RMS_ERR_INVALID_ARG;
    }
    for (int j = i + 1; j < 3; ++j)
      if (overlap(writes[i], write_n[i], writes[j], write_n[j])) return RMS_ERR_INVALID_ARG;
  }
  if (dh && overlap(dh, xb, dy, xb)) return RMS_ERR_INVALID_ARG;

  const bool aligned = (N * b) % 16 == 0 && aligned16(dy) && aligned16(x) && aligned16(gamma) &&
                       aligned16(dx) && (!dh || aligned16(dh));
  BwdArgs a{dy, x, gamma, rstd, dx, dgamma, static_cast<float*>(workspace), M, (int)N,
            (int)dtype, gemma, dh};
  Mapping m;
  float* kbuf = nullptr;
  const rms_status st = plan_bwd(a, path, aligned, d, &m, &kbuf);
  if (st != RMS_OK) return st;
  // The partial rows must fit the workspace before any kernel writes them.
  if ((size_t)m.partials * (size_t)N * sizeof(float) > need) return RMS_ERR_WORKSPACE;

  cudaError_t e;
  switch (m.path) {
    case rmsi::kRegisters:
      e = rmsi::launch_bwd_registers(a, m, s);
      break;
    case rmsi::kStaged:
      e = rmsi::launch_bwd_staged(a, m, d, g_wait_limit.load(), s);
      break;
    case rmsi::kChunked:
      e = rmsi::launch_bwd_chunked(a, m, kbuf, d, g_wait_limit.load(), s);
      if (e == cudaSuccess && !m.wide) g_launches.fetch_add(1);  // three-pass: three kernels
      break;
    default:
      e = rmsi::launch_bwd_scalar(a, m, s);
      break;
  }
  if (e != cudaSuccess) return RMS_ERR_CUDA;
  e = rmsi::launch_colreduce(a.ws, dgamma, m.partials, (int)N, d.sms, s);
  if (e != cudaSuccess) return RMS_ERR_CUDA;
  g_launches.fetch_add(2);
  return RMS_OK;
}

rms_status rms_bwd_ex(void* dy, const void* x, const void* gamma, const float* rstd, void* dx,
                      float* dgamma, void* workspace, size_t workspace_bytes, int64_t M,
                      int64_t N, rms_dtype dtype, int gemma, int inplace_dx, rms_path path,
                      void* stream) {
  return bwd_impl(dy, x, gamma, rstd, nullptr, dx, dgamma, workspace, workspace_bytes, M, N,
                  dtype, gemma, inplace_dx, path, stream);
}

rms_status rms_bwd(void* dy, const void* x, const void* gamma, const float* rstd, void* dx,
                   float* dgamma, void* workspace, int64_t M, int64_t N, rms_dtype dtype, int gemma,
                   int inplace_dx, void* stream) {
  return bwd_impl(dy, x, gamma, rstd, nullptr, dx, dgamma, workspace, SIZE_MAX, M, N, dtype,
                  gemma, inplace_dx, RMS_PATH_AUTO, stream);
}

rms_status rms_bwd_reduction(int64_t M, int64_t N, rms_dtype dtype, int gemma, int residual,
                             rms_path path, int64_t* partials, int64_t* rows_per_partial) {
  if (!partials || !rows_per_partial) return RMS_ERR_INVALID_ARG;
  if (!valid_common(M, N, dtype, gemma)) return RMS_ERR_INVALID_ARG;
  if (residual != 0 && residual != 1) return RMS_ERR_INVALID_ARG;
  if (path < RMS_PATH_AUTO || path > RMS_PATH_CHUNKED) return RMS_ERR_INVALID_ARG;
  if (N > (int64_t)INT32_MAX) return RMS_ERR_UNSUPPORTED;
  *partials = 0;
  *rows_per_partial = 0;
  if (M == 0) return RMS_OK;
  DeviceInfo d;
  if (!current_device(&d)) return RMS_ERR_CUDA;
  // The plan reads only the shape, the types and whether a residual
  // gradient is present (a non-null stand-in; nothing is dereferenced).
  static const char kStandIn = 0;
  BwdArgs a{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, M, (int)N, (int)dtype,
            gemma, residual ? static_cast<const void*>(&kStandIn) : nullptr};
  const bool aligned = (N * elem_bytes(dtype)) % 16 == 0;
  Mapping m;
  float* kbuf = nullptr;
  const rms_status st = plan_bwd(a, path, aligned, d, &m, &kbuf);
  if (st != RMS_OK) return st;
  *partials = m.partials;
  *rows_per_partial = most_rows_per_partial(M, m);
  return RMS_OK;
}

rms_status rms_dgamma_combine(const float* parts, int64_t ranks, int64_t N, float* dgamma,
                              void* stream) {
  if (ranks < 1 || N < 1 || !parts || !dgamma) return RMS_ERR_INVALID_ARG;
  if (ranks > INT64_MAX / N / (int64_t)sizeof(float)) return RMS_ERR_INVALID_ARG;
  if ((N + 3) / 4 > (int64_t)INT32_MAX * 256) return RMS_ERR_UNSUPPORTED;
  if (overlap(dgamma, (size_t)N * sizeof(float), parts, (size_t)(ranks * N) * sizeof(float)))
    return RMS_ERR_INVALID_ARG;
  if (rmsi::launch_rank_sum(parts, dgamma, ranks, N, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return RMS_ERR_CUDA;
  g_launches.fetch_add(1);
  return RMS_OK;
}

rms_status rms_dgamma_cast(const float* dgamma, void* out, int64_t N, rms_dtype dtype,
                           void* stream) {
  if (N < 1 || !dgamma || !out) return RMS_ERR_INVALID_ARG;
  if (dtype < RMS_F32 || dtype > RMS_F16_W32) return RMS_ERR_INVALID_ARG;
  if ((N + 3) / 4 > (int64_t)INT32_MAX * 256) return RMS_ERR_UNSUPPORTED;
  const size_t wb = (size_t)rmsi::weight_bytes(dtype);
  if (overlap(out, (size_t)N * wb, dgamma, (size_t)N * sizeof(float))) return RMS_ERR_INVALID_ARG;
  if (rmsi::launch_weight_cast(dgamma, out, N, dtype, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return RMS_ERR_CUDA;
  g_launches.fetch_add(1);
  return RMS_OK;
}

rms_status rms_fwd_quant_ex(const void* x, const void* gamma, uint8_t* q, float* scale,
                            float* rstd, int64_t M, int64_t N, float eps, rms_dtype dtype,
                            int gemma, rms_path path, void* stream) {
  if (!valid_common(M, N, dtype, gemma)) return RMS_ERR_INVALID_ARG;
  if (!isfinite(eps) || eps < 0.f) return RMS_ERR_INVALID_ARG;
  if (path < RMS_PATH_AUTO || path > RMS_PATH_CHUNKED) return RMS_ERR_INVALID_ARG;
  if (path == RMS_PATH_STAGED) return RMS_ERR_UNSUPPORTED;
  if (N > (int64_t)INT32_MAX) return RMS_ERR_UNSUPPORTED;
  if (M == 0) return RMS_OK;
  if (!x || !gamma || !q || !scale || !rstd) return RMS_ERR_INVALID_ARG;
  const int b = elem_bytes(dtype);
  const size_t xb = matrix_bytes(M, N, b);
  const size_t qb = matrix_bytes(M, N, 1);
  if (xb == 0 || qb == 0) return RMS_ERR_INVALID_ARG;
  const size_t gb = (size_t)N * rmsi::weight_bytes(dtype), rb = (size_t)M * sizeof(float);
  const void* reads[2] = {x, gamma};
  const size_t read_n[2] = {xb, gb};
  const void* writes[3] = {q, scale, rstd};
  const size_t write_n[3] = {qb, rb, rb};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 2; ++j)
      if (overlap(writes[i], write_n[i], reads[j], read_n[j])) return RMS_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (overlap(writes[i], write_n[i], writes[j], write_n[j])) return RMS_ERR_INVALID_ARG;
  }
  DeviceInfo d;
  if (!current_device(&d)) return RMS_ERR_CUDA;
  const bool aligned =
      (N * b) % 16 == 0 && aligned16(x) && aligned16(gamma) && aligned16(q);
  Mapping m;
  if ((path == RMS_PATH_REGISTERS || path == RMS_PATH_CHUNKED) && !aligned)
    return RMS_ERR_ALIGNMENT;
  const bool regs = aligned && rmsi::plan_quant_registers((int)N, dtype, &m);
  bool wide = false;
  if (path == RMS_PATH_REGISTERS && !regs) return RMS_ERR_UNSUPPORTED;
  if (path == RMS_PATH_SCALAR || !aligned) {
    if (M > INT32_MAX) return RMS_ERR_UNSUPPORTED;
    m.path = rmsi::kScalar;
  } else if (path == RMS_PATH_CHUNKED || !regs) {
    // aligned rows too wide for the registers: one pass in a cluster of CTAs
    // while the row's slices fit, else a CTA per row walking it three times
    Mapping mw;
    if (rmsi::plan_quant_wide((int)N, dtype, &mw)) {
      wide = true;
      m = mw;
    } else {
      if (M > INT32_MAX) return RMS_ERR_UNSUPPORTED;
      m.path = rmsi::kChunked;
    }
  } else if ((M + m.rows_per_cta - 1) / m.rows_per_cta > INT32_MAX) {
    return RMS_ERR_UNSUPPORTED;
  }
  rmsi::QuantArgs a{x, gamma, q, scale, rstd, M, (int)N, eps, (int)dtype, gemma};
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = wide ? rmsi::launch_fwd_quant_wide(a, m, d, g_wait_limit.load(), s)
                             : rmsi::launch_fwd_quant(a, m, s);
  if (e != cudaSuccess) return RMS_ERR_CUDA;
  g_launches.fetch_add(1);
  return RMS_OK;
}

rms_status rms_fwd_quant(const void* x, const void* gamma, uint8_t* q, float* scale, float* rstd,
                         int64_t M, int64_t N, float eps, rms_dtype dtype, int gemma,
                         void* stream) {
  return rms_fwd_quant_ex(x, gamma, q, scale, rstd, M, N, eps, dtype, gemma, RMS_PATH_AUTO,
                          stream);
}

rms_status rms_bwd_add_ex(void* dy, const void* h, const void* gamma, const float* rstd,
                          const void* dh, void* dx, float* dgamma, void* workspace,
                          size_t workspace_bytes, int64_t M, int64_t N, rms_dtype dtype,
                          int gemma, int inplace_dx, rms_path path, void* stream) {
  if (M > 0 && !dh) return RMS_ERR_INVALID_ARG;
  return bwd_impl(dy, h, gamma, rstd, dh, dx, dgamma, workspace, workspace_bytes, M, N, dtype,
                  gemma, inplace_dx, path, stream);
}

rms_status rms_bwd_add(void* dy, const void* h, const void* gamma, const float* rstd,
                       const void* dh, void* dx, float* dgamma, void* workspace, int64_t M,
                       int64_t N, rms_dtype dtype, int gemma, int inplace_dx, void* stream) {
  return rms_bwd_add_ex(dy, h, gamma, rstd, dh, dx, dgamma, workspace, SIZE_MAX, M, N, dtype,
                        gemma, inplace_dx, RMS_PATH_AUTO, stream);
}

rms_status rms_last_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return RMS_ERR_CUDA;
  int v = 0, w = 0, c = 0;
  if (rmsi::take_device_status(&v) != cudaSuccess) return RMS_ERR_CUDA;
  if (rmsi::take_ln_device_status(&w) != cudaSuccess) return RMS_ERR_CUDA;
  if (rmsi::take_wide_device_status(&c) != cudaSuccess) return RMS_ERR_CUDA;
  return (v || w || c) ? RMS_ERR_TIMEOUT : RMS_OK;
}

size_t ln_bwd_workspace_size(int64_t M, int64_t N) {
  if (M <= 0 || N <= 0) return 0;
  DeviceInfo d;
  if (!current_device(&d)) return 0;
  return 2 * workspace_need(M, N, d);
}

rms_status ln_fwd_ex(const void* x, const void* w, const void* b, void* y, float* mean,
                     float* rstd, int64_t M, int64_t N, float eps, rms_dtype dtype, rms_path path,
                     void* stream) {
  if (!valid_common(M, N, dtype, 0)) return RMS_ERR_INVALID_ARG;
  if (!isfinite(eps) || eps < 0.f) return RMS_ERR_INVALID_ARG;
  if (path < RMS_PATH_AUTO || path > RMS_PATH_CHUNKED) return RMS_ERR_INVALID_ARG;
  if (path == RMS_PATH_STAGED || path == RMS_PATH_CHUNKED) return RMS_ERR_UNSUPPORTED;
  if (N > (int64_t)INT32_MAX) return RMS_ERR_UNSUPPORTED;
  if (M == 0) return RMS_OK;
  if (!x || !w || !y || !mean || !rstd) return RMS_ERR_INVALID_ARG;
  const int bsz = elem_bytes(dtype);
  const size_t xb = matrix_bytes(M, N, bsz);
  if (xb == 0) return RMS_ERR_INVALID_ARG;
  const size_t wb = (size_t)N * rmsi::weight_bytes(dtype), rb = (size_t)M * sizeof(float);
  const void* reads[3] = {x, w, b};
  const size_t read_n[3] = {xb, wb, wb};
  const void* writes[3] = {y, mean, rstd};
  const size_t write_n[3] = {xb, rb, rb};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 3; ++j)
      if (overlap(writes[i], write_n[i], reads[j], read_n[j])) return RMS_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (overlap(writes[i], write_n[i], writes[j], write_n[j])) return RMS_ERR_INVALID_ARG;
  }
  DeviceInfo d;
  if (!current_device(&d)) return RMS_ERR_CUDA;
  const bool aligned = (N * bsz) % 16 == 0 && aligned16(x) && aligned16(w) && aligned16(y) &&
                       (!b || aligned16(b));
  Mapping m;
  if (path == RMS_PATH_REGISTERS && !aligned) return RMS_ERR_ALIGNMENT;
  if (!rmsi::ln_plan((int)N, dtype, false, path, aligned, d, &m)) return RMS_ERR_UNSUPPORTED;
  if (m.path == rmsi::kScalar && M > INT32_MAX) return RMS_ERR_UNSUPPORTED;
  if (m.path == rmsi::kRegisters && (M + m.rows_per_cta - 1) / m.rows_per_cta > INT32_MAX)
    return RMS_ERR_UNSUPPORTED;
  rmsi::LnFwdArgs a{x, w, b, y, mean, rstd, M, (int)N, eps, (int)dtype};
  if (rmsi::ln_launch_fwd(a, m, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return RMS_ERR_CUDA;
  g_launches.fetch_add(1);
  return RMS_OK;
}

rms_status ln_fwd(const void* x, const void* w, const void* b, void* y, float* mean, float* rstd,
                  int64_t M, int64_t N, float eps, rms_dtype dtype, void* stream) {
  return ln_fwd_ex(x, w, b, y, mean, rstd, M, N, eps, dtype, RMS_PATH_AUTO, stream);
}

rms_status ln_bwd_ex(void* dy, const void* x, const void* w, const float* mean,
                     const float* rstd, void* dx, float* dw, float* db, void* workspace,
                     size_t workspace_bytes, int64_t M, int64_t N, rms_dtype dtype, int inplace_dx,
                     rms_path path, void* stream) {
  if (!valid_common(M, N, dtype, 0)) return RMS_ERR_INVALID_ARG;
  if (inplace_dx != 0 && inplace_dx != 1) return RMS_ERR_INVALID_ARG;
  if (path < RMS_PATH_AUTO || path > RMS_PATH_CHUNKED) return RMS_ERR_INVALID_ARG;
  if (path == RMS_PATH_REGISTERS || path == RMS_PATH_CHUNKED) return RMS_ERR_UNSUPPORTED;
  if (N > (int64_t)INT32_MAX) return RMS_ERR_UNSUPPORTED;
  if (inplace_dx) {
    if (dx && dx != dy) return RMS_ERR_INVALID_ARG;
    dx = dy;
  }
  if (!dw) return RMS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 0) {
    if (cudaMemsetAsync(dw, 0, (size_t)N * sizeof(float), s) != cudaSuccess) return RMS_ERR_CUDA;
    if (db && cudaMemsetAsync(db, 0, (size_t)N * sizeof(float), s) != cudaSuccess)
      return RMS_ERR_CUDA;
    return RMS_OK;
  }
  if (!dx || !dy || !x || !w || !mean || !rstd) return RMS_ERR_INVALID_ARG;
  if (!workspace) return RMS_ERR_WORKSPACE;
  const int bsz = elem_bytes(dtype);
  const size_t xb = matrix_bytes(M, N, bsz);
  if (xb == 0) return RMS_ERR_INVALID_ARG;
  DeviceInfo d;
  if (!current_device(&d)) return RMS_ERR_CUDA;
  const size_t half = workspace_need(M, N, d);
  if (workspace_bytes < 2 * half || ((uintptr_t)workspace & 255u) != 0) return RMS_ERR_WORKSPACE;
  const size_t wb = (size_t)N * rmsi::weight_bytes(dtype), rb = (size_t)M * sizeof(float),
               vb = (size_t)N * sizeof(float);
  const void* reads[5] = {dy, x, w, mean, rstd};
  const size_t read_n[5] = {xb, xb, wb, rb, rb};
  const void* writes[4] = {dx, dw, db, workspace};
  const size_t write_n[4] = {xb, vb, vb, 2 * half};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 5; ++j) {
      if (i == 0 && j == 0 && dx == dy) continue;  // the sanctioned in-place alias
      if (overlap(writes[i], write_n[i], reads[j], read_n[j])) return RMS_ERR_INVALID_ARG;
    }
    for (int j = i + 1; j < 4; ++j)
      if (overlap(writes[i], write_n[i], writes[j], write_n[j])) return RMS_ERR_INVALID_ARG;
  }
  const bool aligned = (N * bsz) % 16 == 0 && aligned16(dy) && aligned16(x) && aligned16(w) &&
                       aligned16(dx);
  if (path == RMS_PATH_STAGED && !aligned) return RMS_ERR_ALIGNMENT;
  Mapping m;
  if (!rmsi::ln_plan((int)N, dtype, true, path, aligned, d, &m, M)) return RMS_ERR_UNSUPPORTED;
  float* wsw = static_cast<float*>(workspace);
  float* wsb = reinterpret_cast<float*>(static_cast<char*>(workspace) + half);
  rmsi::LnBwdArgs a{dy, x, w, mean, rstd, dx, wsw, wsb, M, (int)N, (int)dtype};
  if (rmsi::ln_size_bwd(a, d, &m) != cudaSuccess) return RMS_ERR_CUDA;
  // The partial rows must fit the workspace before any kernel writes them.
  if ((size_t)m.partials * (size_t)N * sizeof(float) > half) return RMS_ERR_WORKSPACE;
  if (rmsi::ln_launch_bwd(a, m, g_wait_limit.load(), s) != cudaSuccess) return RMS_ERR_CUDA;
  // dw and db: one launch when both are vectorisable, else one each
  if (rmsi::launch_colreduce2(wsw, dw, db ? wsb : nullptr, db, m.partials, (int)N, d.sms, s) !=
      cudaSuccess)
    return RMS_ERR_CUDA;
  const bool vec = N % 4 == 0 && aligned16(dw) && (!db || aligned16(db));
  g_launches.fetch_add(db && !vec ? 3 : 2);
  return RMS_OK;
}

rms_status ln_bwd_reduction(int64_t M, int64_t N, rms_dtype dtype, rms_path path,
                            int64_t* partials, int64_t* rows_per_partial) {
  if (!partials || !rows_per_partial) return RMS_ERR_INVALID_ARG;
  if (!valid_common(M, N, dtype, 0)) return RMS_ERR_INVALID_ARG;
  if (path < RMS_PATH_AUTO || path > RMS_PATH_CHUNKED) return RMS_ERR_INVALID_ARG;
  if (path == RMS_PATH_REGISTERS || path == RMS_PATH_CHUNKED) return RMS_ERR_UNSUPPORTED;
  if (N > (int64_t)INT32_MAX) return RMS_ERR_UNSUPPORTED;
  *partials = 0;
  *rows_per_partial = 0;
  if (M == 0) return RMS_OK;
  DeviceInfo d;
  if (!current_device(&d)) return RMS_ERR_CUDA;
  const bool aligned = (N * elem_bytes(dtype)) % 16 == 0;
  if (path == RMS_PATH_STAGED && !aligned) return RMS_ERR_ALIGNMENT;
  Mapping m;
  if (!rmsi::ln_plan((int)N, dtype, true, path, aligned, d, &m, M)) return RMS_ERR_UNSUPPORTED;
  rmsi::LnBwdArgs a{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                    M, (int)N, (int)dtype};
  if (rmsi::ln_size_bwd(a, d, &m) != cudaSuccess) return RMS_ERR_CUDA;
  *partials = m.partials;
  *rows_per_partial = most_rows_per_partial(M, m);
  return RMS_OK;
}

rms_status ln_bwd(void* dy, const void* x, const void* w, const float* mean, const float* rstd,
                  void* dx, float* dw, float* db, void* workspace, int64_t M, int64_t N,
                  rms_dtype dtype, int inplace_dx, void* stream) {
  return ln_bwd_ex(dy, x, w, mean, rstd, dx, dw, db, workspace, SIZE_MAX, M, N, dtype, inplace_dx,
                   RMS_PATH_AUTO, stream);
}

}  // extern "C"
