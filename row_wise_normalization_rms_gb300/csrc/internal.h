// Host-side interface between the C ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace rmsi {

// Element types of a call: activations (x, y, dy, dx) and weight (gamma).
enum Dtype { kF32 = 0, kBF16 = 1, kF16 = 2, kBF16W32 = 3, kF16W32 = 4 };

// Bytes of one activation element / one weight element.
inline int dtype_bytes(int dtype) { return dtype == kF32 ? 4 : 2; }
inline int weight_bytes(int dtype) { return (dtype == kBF16 || dtype == kF16) ? 2 : 4; }
enum Path { kAuto = 0, kRegisters = 1, kStaged = 2, kScalar = 3, kChunked = 4 };

struct FwdArgs {
  const void* x;
  const void* gamma;
  void* y;
  float* rstd;
  int64_t M;
  int N;
  float eps;
  int dtype;
  int gemma;
  const void* res = nullptr;  // fused residual add: the row is h = x + res ...
  void* h = nullptr;          // ... stored here (may equal res)
};

struct BwdArgs {
  void* dy;
  const void* x;
  const void* gamma;
  const float* rstd;
  void* dx;  // == dy for in-place dx
  float* dgamma;
  float* ws;  // [P][N] float32 column partials
  int64_t M;
  int N;
  int dtype;
  int gemma;
  const void* dh = nullptr;  // fused residual add: dx += dh (may equal dx)
};

// How one launch maps rows onto the GPU.
struct Mapping {
  int path = kAuto;
  int G = 0;             // threads per row
  int kv = 0;            // 16-byte vectors per thread per row (register path)
  int threads = 0;       // threads per CTA
  int rows_per_cta = 0;  // rows a CTA works on at once (threads / G)
  int64_t blocks = 0;    // CTAs launched
  int64_t partials = 0;  // backward: workspace rows of column partials (one per CTA or cluster)
  int stages = 0;        // shared-memory pipeline depth (staged path)
  int cluster = 1;       // CTAs per cluster sharing one row (staged path)
  int sv = 0;            // 16-byte vectors per CTA's column slice (staged path)
  int smem_acc = 0;      // scalar backward: partials in shared memory (else in the workspace)
  int chunks = 0;        // chunked path: chunks per row
  int wide = 0;          // chunked path: one pass over memory, a cluster of CTAs per row
  size_t smem = 0;       // dynamic shared memory bytes
};

struct DeviceInfo {
  int device = 0;
  int sms = 0;
  size_t smem_optin = 0;  // max dynamic shared memory per CTA
};

// Raises a kernel's dynamic shared memory limit to the device maximum
// (once per kernel and device; thread-safe).  Defined in api.cu.
cudaError_t opt_in_max_smem(const void* kernel, const DeviceInfo& d);

// Largest number of persistent CTAs a backward launch may use on a device
// with `sms` SMs; the workspace holds this many float32 rows of N.
inline int64_t max_partials(int sms) { return 4 * (int64_t)sms; }

// ---- register path (fwd_registers.cu, bwd_registers.cu) ----
bool plan_registers(int N, int dtype, bool bwd, Mapping* m);
cudaError_t launch_fwd_registers(const FwdArgs& a, const Mapping& m, cudaStream_t s);
// Fill m.blocks (CTAs) and m.partials (workspace rows) for a persistent backward.
cudaError_t size_bwd_registers(const BwdArgs& a, const DeviceInfo& d, Mapping* m);
cudaError_t launch_bwd_registers(const BwdArgs& a, const Mapping& m, cudaStream_t s);

// ---- scalar path and the column reduction (scalar.cu) ----
bool plan_scalar(int N, int dtype, bool bwd, const DeviceInfo& d, Mapping* m);
cudaError_t launch_fwd_scalar(const FwdArgs& a, const Mapping& m, cudaStream_t s);
cudaError_t size_bwd_scalar(const BwdArgs& a, const DeviceInfo& d, Mapping* m);
cudaError_t launch_bwd_scalar(const BwdArgs& a, const Mapping& m, cudaStream_t s);
// dgamma[j] = sum_{p < P} ws[p][j] in a fixed order that depends on P and N
// only (bitwise reproducible); sms sizes the grid.
cudaError_t launch_colreduce(const float* ws, float* dgamma, int64_t P, int N, int sms,
                             cudaStream_t s);
// Two such sums (out0 from ws0, out1 from ws1) in one launch; ws1 == NULL
// makes it the single sum.
cudaError_t launch_colreduce2(const float* ws0, float* out0, const float* ws1, float* out1,
                              int64_t P, int N, int sms, cudaStream_t s);
// out[j] = sum over r < R of parts[r][j], added in increasing r.
cudaError_t launch_rank_sum(const float* parts, float* out, int64_t R, int64_t N, cudaStream_t s);
// dst[j] = src[j] in the weight type of `dtype` (bf16 / fp16 rounded to
// nearest even; float32 copied).
cudaError_t launch_weight_cast(const float* src, void* dst, int64_t N, int dtype, cudaStream_t s);

// ---- chunked path: rows of any width (chunked.cu) ----
bool plan_chunked(int N, int dtype, bool bwd, bool res, Mapping* m);
cudaError_t launch_fwd_chunked(const FwdArgs& a, const Mapping& m, const DeviceInfo& d,
                               long long wait_limit, cudaStream_t s);
// Fill m.blocks and m.partials and choose where the per-row k values live;
// false when the shape leaves no room for them in the workspace.
bool size_bwd_chunked(const BwdArgs& a, const DeviceInfo& d, Mapping* m, float** kbuf);
cudaError_t launch_bwd_chunked(const BwdArgs& a, const Mapping& m, float* kbuf,
                               const DeviceInfo& d, long long wait_limit, cudaStream_t s);
// Reads and clears the one-pass kernels' device status word (nonzero: an
// exchange wait ran past the wait limit).
cudaError_t take_wide_device_status(int* status);

// ---- forward with the output quantised to FP8 E4M3 (quant.cu) ----
struct QuantArgs {
  const void* x;
  const void* gamma;
  uint8_t* q;     // [M][N] E4M3 codes
  float* scale;   // [M] per-row scale: y ~ code * scale
  float* rstd;    // [M]
  int64_t M;
  int N;
  float eps;
  int dtype;
  int gemma;
};
// m.path kRegisters (plan_registers), kChunked (aligned rows of any width:
// a CTA per row) or kScalar.
// The register mapping of the E4M3 forward (rows up to 32 KiB).
bool plan_quant_registers(int N, int dtype, Mapping* m);
cudaError_t launch_fwd_quant(const QuantArgs& a, const Mapping& m, cudaStream_t s);
// Rows too wide for the registers whose slices of 4 x 512 vectors number at
// most 16: a cluster of CTAs per row, one pass over HBM (chunked.cu).  false
// when the row needs more slices.
bool plan_quant_wide(int N, int dtype, Mapping* m);
cudaError_t launch_fwd_quant_wide(const QuantArgs& a, const Mapping& m, const DeviceInfo& d,
                                  long long wait_limit, cudaStream_t s);

// ---- LayerNorm (layernorm.cu) ----
struct LnFwdArgs {
  const void* x;
  const void* w;
  const void* b;  // may be null: no bias
  void* y;
  float* mean;
  float* rstd;
  int64_t M;
  int N;
  float eps;
  int dtype;
};

struct LnBwdArgs {
  const void* dy;
  const void* x;
  const void* w;
  const float* mean;
  const float* rstd;
  void* dx;   // == dy for in-place dx
  float* wsw;  // [P][N] dw partials
  float* wsb;  // [P][N] db partials
  int64_t M;
  int N;
  int dtype;
};

// Chooses the LayerNorm mapping for a call (path as rms_path); false when
// the requested path cannot take the shape.
bool ln_plan(int N, int dtype, bool bwd, int path, bool aligned, const DeviceInfo& d, Mapping* m,
             int64_t M = 0);
cudaError_t ln_launch_fwd(const LnFwdArgs& a, const Mapping& m, cudaStream_t s);
cudaError_t ln_size_bwd(const LnBwdArgs& a, const DeviceInfo& d, Mapping* m);
cudaError_t ln_launch_bwd(const LnBwdArgs& a, const Mapping& m, long long wait_limit,
                          cudaStream_t s);
cudaError_t take_ln_device_status(int* status);

// ---- staged path (staged.cu) ----
// res: the fused residual add stages one more tensor (the residual, or dh).
// M (0: unknown) lets the plan shorten tiles when few rows would leave the
// persistent CTAs' last wave ragged.
bool plan_staged(int N, int dtype, bool bwd, const DeviceInfo& d, Mapping* m, bool res = false,
                 int64_t M = 0);
cudaError_t launch_fwd_staged(const FwdArgs& a, const Mapping& m, const DeviceInfo& d,
                              long long wait_limit, cudaStream_t s);
cudaError_t size_bwd_staged(const BwdArgs& a, const DeviceInfo& d, Mapping* m);
cudaError_t launch_bwd_staged(const BwdArgs& a, const Mapping& m, const DeviceInfo& d,
                              long long wait_limit, cudaStream_t s);
// Reads and clears the device status word of the current device
// (0 = no bounded wait gave up since the last call).
cudaError_t take_device_status(int* status);

}  // namespace rmsi
