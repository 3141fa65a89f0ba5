/*
 * rmsnorm.h — C ABI of the GB300 (sm_103a) fused RMSNorm library
 * (librmsnorm.so).
 *
 * What it computes, per row i of an M x N row-major matrix, with
 * g_j = gamma_j, or 1 + gamma_j in Gemma mode:
 *
 *   forward   r_i  = 1 / sqrt( (1/N) sum_j x_ij^2 + eps )
 *             y_ij = x_ij * r_i * g_j
 *   backward  u_ij = dy_ij * g_j
 *             c_i  = (1/N) sum_j u_ij * x_ij
 *             dx_ij = r_i * u_ij - x_ij * r_i^3 * c_i
 *             dgamma_j = sum_i dy_ij * x_ij * r_i      (a sum over rows)
 *
 * Sources: "Hướng dẫn Triton RMSNorm: kernel, backward…" (partitech.com),
 * sections "Vấn đề và công thức tham chiếu" (forward, eps under the square
 * root), "Vì sao cần một lượt đi và một lượt về?" (backward formulas),
 * "N và BLOCK: hai kích thước không được nhầm" (the mean divides by the true
 * N), "Reduce dgamma không có race khi ghi" and "Tổng không phải trung bình"
 * (dgamma as per-part partial sums reduced in a second pass; a sum, not a
 * mean); "02 · 手写 Triton kernel:RMSNorm / RoPE / SwiGLU", section 3
 * (Gemma's (1 + W) weight, the cast of the normalised row to the weight
 * dtype before the weight multiply, dx written into dy's buffer).
 *
 * Conventions shared by every entry point
 *  - Every tensor argument is a DEVICE pointer owned by the caller.  The
 *    library allocates nothing and keeps no per-call state; all work is
 *    enqueued asynchronously on `stream` (a cudaStream_t passed as void*;
 *    NULL selects the legacy default stream of the current device).
 *  - Matrices are contiguous row-major with row stride N elements.
 *    x, y, dy, dx share the activation type of `dtype`, gamma its weight
 *    type (see rms_dtype).  rstd is always float32 (M entries), dgamma
 *    always float32 (N entries).
 *  - Arithmetic is float32 throughout (loads widened to float32, float32
 *    accumulation, one rounding to `dtype` per stored element), except the
 *    non-Gemma low-precision forward, which rounds x*r to `dtype` before
 *    multiplying by gamma (the cast order of the source above).
 *  - Pointers that are not 16-byte aligned, or N*sizeof(dtype) not a
 *    multiple of 16, select a slower scalar path; they are not an error.
 *  - Arguments are validated on the host before anything is launched.  On
 *    any error nothing is enqueued and the status says why.  No CPU
 *    fallback exists: unsupported shapes are rejected.
 */
#ifndef RMSNORM_H_
#define RMSNORM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of a call.  The first three use one type for activations
 * (x, y, dy, dx) and weight (gamma); the _W32 codes pair 16-bit activations
 * with a float32 gamma (the normalised row is then "cast" to float32, which
 * is exact, and y is one rounding of x*r*gamma). */
typedef enum {
  RMS_F32 = 0,      /* IEEE float32 */
  RMS_BF16 = 1,     /* bfloat16 (8-bit significand), round-to-nearest-even on store */
  RMS_F16 = 2,      /* IEEE float16 (11-bit significand), round-to-nearest-even on store */
  RMS_BF16_W32 = 3, /* bfloat16 activations, float32 gamma */
  RMS_F16_W32 = 4   /* float16 activations, float32 gamma */
} rms_dtype;

typedef enum {
  RMS_OK = 0,
  RMS_ERR_INVALID_ARG = 1, /* null pointer, bad size, eps, flag, dtype, or overlapping buffers */
  RMS_ERR_UNSUPPORTED = 2, /* N too large for every row mapping on this device */
  RMS_ERR_ALIGNMENT = 3,   /* an explicitly requested path needs 16-byte aligned rows */
  RMS_ERR_WORKSPACE = 4,   /* workspace missing or smaller than rms_bwd_workspace_size() */
  RMS_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
  RMS_ERR_TIMEOUT = 6      /* a device-side bounded wait gave up (see rms_last_device_status) */
} rms_status;

/* Row mapping, for rms_fwd_ex / rms_bwd_ex.  RMS_PATH_AUTO picks from N and
 * dtype; the others force one mapping (used to test and time each). */
typedef enum {
  RMS_PATH_AUTO = 0,
  RMS_PATH_REGISTERS = 1, /* a warp or a thread group per row, row held in registers */
  RMS_PATH_STAGED = 2,    /* persistent CTAs, rows staged in shared memory by cp.async.bulk */
  RMS_PATH_SCALAR = 3,    /* element-wise loads, any alignment */
  RMS_PATH_CHUNKED = 4    /* any width, RMSNorm only: rows of up to 16 slices (forward
                             16 x 128 KiB, backward 16 x 32 KiB) go through a cluster of
                             CTAs in one pass over memory; wider rows take three passes (a
                             row pass, then the outputs from a second read).  Chosen by
                             RMS_PATH_AUTO for rows the others split over a cluster or
                             cannot take.  rms_fwd_quant: rows of up to 16 x 32 KiB in
                             one pass through a cluster, a CTA per row beyond */
} rms_path;

/*
 * rms_fwd — forward RMSNorm over M rows of N.
 *   x     [M*N] dtype, read.
 *   gamma [N]   dtype, read (the weight; used as 1+gamma when gemma=1).
 *   y     [M*N] dtype, written.  Must not overlap x, gamma or rstd.
 *   rstd  [M]   float32, written: r_i, kept for rms_bwd.
 *   M >= 0 (M == 0 is a no-op), N >= 1, eps finite and >= 0, gemma in {0,1}.
 * Source: the forward formula and worked example of "Hướng dẫn Triton
 * RMSNorm", section "Vấn đề và công thức tham chiếu"; Gemma weight and cast
 * order from "02 · 手写 Triton kernel", section 3.
 * Errors: RMS_ERR_INVALID_ARG, RMS_ERR_UNSUPPORTED, RMS_ERR_CUDA.  With
 * eps == 0 an all-zero row gives r = +inf and y = NaN (no special case).
 */
rms_status rms_fwd(const void* x, const void* gamma, void* y, float* rstd,
                   int64_t M, int64_t N, float eps, rms_dtype dtype, int gemma,
                   void* stream);

/* rms_fwd with an explicit row mapping (see rms_path).  A forced mapping
 * that cannot run the shape returns RMS_ERR_UNSUPPORTED or
 * RMS_ERR_ALIGNMENT instead of falling back. */
rms_status rms_fwd_ex(const void* x, const void* gamma, void* y, float* rstd,
                      int64_t M, int64_t N, float eps, rms_dtype dtype, int gemma,
                      rms_path path, void* stream);

/*
 * rms_bwd — backward RMSNorm: dx and dgamma from dy, x, gamma and the rstd
 * the forward saved (eps enters only through rstd, which is used as given).
 *   dy     [M*N] dtype, read; overwritten with dx when inplace_dx = 1.
 *   x      [M*N] dtype, read.      gamma [N] dtype, read.
 *   rstd   [M]   float32, read.
 *   dx     [M*N] dtype, written.  With inplace_dx = 1 it must be NULL or
 *          equal to dy, and dx is written into dy's buffer.
 *   dgamma [N]   float32, written: sum over rows of dy*x*r (no mean).
 *   workspace  device scratch of at least rms_bwd_workspace_size(M, N)
 *          bytes, 256-byte aligned, owned by the caller; holds one float32
 *          row of column partial sums per persistent CTA.  Contents on entry
 *          are ignored, on return undefined.  May be NULL only when M == 0.
 *   dtype, gemma in {0,1}, inplace_dx in {0,1} as for rms_fwd.
 * dgamma is computed in two deterministic stages (per-CTA partials over a
 * static row assignment, then a fixed-order column sum; no atomics, no
 * locks), so it is bitwise identical from run to run on one device.
 * Written buffers must not overlap any other argument (except dx == dy
 * with inplace_dx = 1).  M == 0 writes dgamma = 0.
 * Source: the backward formulas of "Hướng dẫn Triton RMSNorm", sections
 * "Vì sao cần một lượt đi và một lượt về?", "Backward đầu vào: giữ đúng N",
 * "Reduce dgamma không có race khi ghi", "Tổng không phải trung bình";
 * in-place dx from "02 · 手写 Triton kernel", section 3.
 * Errors: RMS_ERR_INVALID_ARG, RMS_ERR_UNSUPPORTED, RMS_ERR_WORKSPACE,
 * RMS_ERR_CUDA.
 */
rms_status rms_bwd(void* dy, const void* x, const void* gamma, const float* rstd,
                   void* dx, float* dgamma, void* workspace,
                   int64_t M, int64_t N, rms_dtype dtype, int gemma, int inplace_dx,
                   void* stream);

/* rms_bwd with the workspace size stated (checked against the need:
 * RMS_ERR_WORKSPACE when too small) and an explicit row mapping.  With
 * RMS_PATH_CHUNKED on rows over 16 slices (the three-pass form) the per-row
 * values between its passes are kept in dgamma when M <= N, else in the
 * workspace's last rows; RMS_ERR_UNSUPPORTED when M > N and they do not fit
 * beside the partial rows. */
rms_status rms_bwd_ex(void* dy, const void* x, const void* gamma, const float* rstd,
                      void* dx, float* dgamma, void* workspace, size_t workspace_bytes,
                      int64_t M, int64_t N, rms_dtype dtype, int gemma, int inplace_dx,
                      rms_path path, void* stream);

/*
 * rms_bwd_reduction — how rms_bwd (residual = 0) or rms_bwd_add
 * (residual = 1) sums dgamma for M rows of N on the current device, so that
 * a caller can bound its float32 rounding error.  The mapping is the one
 * the call would take with 16-byte aligned pointers, or the one `path`
 * forces.
 *   *partials          P: the float32 partial rows the backward writes to
 *                      its workspace; the column sum adds these P values
 *                      per column in a fixed order.
 *   *rows_per_partial  the most rows whose terms dy*x*r any one partial row
 *                      sums (in a fixed order).
 * Any fixed order of float32 additions of n terms carries each term through
 * at most n - 1 roundings, so with u = 2^-24 and D = rows_per_partial + P:
 *   |dgamma_j - sum_i t_ij| <= (D u / (1 - D u)) sum_i |t_ij|,
 * t_ij being each term as the kernel forms it (x*r rounded once, times dy).
 * Both are 0 for M == 0.  Launches nothing.
 * Source: "Hướng dẫn Triton RMSNorm", section "Reduce dgamma không có race
 * khi ghi" (per-part partial sums, then a second pass over the partials).
 * Errors: RMS_ERR_INVALID_ARG (null outputs, bad shape, dtype, flag or
 * path), RMS_ERR_ALIGNMENT / RMS_ERR_UNSUPPORTED as the forced mapping
 * would return them, RMS_ERR_CUDA (device query failed).
 */
rms_status rms_bwd_reduction(int64_t M, int64_t N, rms_dtype dtype, int gemma, int residual,
                             rms_path path, int64_t* partials, int64_t* rows_per_partial);

/*
 * rms_dgamma_combine — the exchange step of a row-sharded backward: each of
 * `ranks` processes ran rms_bwd on its own contiguous block of rows and
 * gathered every rank's dgamma; the total is
 *   dgamma_j = parts[0][j] + parts[1][j] + ... + parts[ranks-1][j]
 * added in increasing rank order, one float32 rounding per addition, so
 * every rank computes the same bits whatever order the gather used.
 *   parts   [ranks][N] float32, read (row r: rank r's dgamma).
 *   dgamma  [N] float32, written; must not overlap parts.
 * Source: "Hướng dẫn Triton RMSNorm", section "Tổng không phải trung bình"
 * (dgamma is a sum over all rows, so per-part sums add up to it) and
 * "Reduce dgamma không có race khi ghi" (partial sums reduced in a fixed
 * second pass, no atomics).
 * Errors: RMS_ERR_INVALID_ARG (null pointer, ranks < 1, N < 1, overlap),
 * RMS_ERR_CUDA.
 */
rms_status rms_dgamma_combine(const float* parts, int64_t ranks, int64_t N, float* dgamma,
                              void* stream);

/*
 * rms_dgamma_cast — the float32 weight gradient handed back in the weight's
 * own type, as the framework wrapper of the source does after its float32
 * column sum: out_j = dgamma_j rounded to nearest (ties to even) in the
 * weight type of `dtype` (bfloat16 for RMS_BF16, float16 for RMS_F16; a
 * float32 copy for RMS_F32, RMS_BF16_W32 and RMS_F16_W32, whose weight is
 * float32).  Works for any float32 N-vector: rms_bwd's dgamma, the total of
 * rms_dgamma_combine, ln_bwd's dw or db.  Values beyond the type's range
 * round to infinity (bfloat16 and float16 have no saturating cast here).
 *   dgamma  [N] float32, read.
 *   out     [N] weight type, written; must not overlap dgamma.
 * The sums stay float32 everywhere else in the library; this is the one
 * optional rounding to the weight type.
 * Source: "Hướng dẫn Triton RMSNorm", section "Reduce dgamma không có race
 * khi ghi" (the partial sums are reduced in float32 and the result cast to
 * the weight's dtype by the backward wrapper).
 * Errors: RMS_ERR_INVALID_ARG (null pointer, N < 1, dtype, overlap),
 * RMS_ERR_CUDA.
 */
rms_status rms_dgamma_cast(const float* dgamma, void* out, int64_t N, rms_dtype dtype,
                           void* stream);

/*
 * rms_bwd_noalloc — rms_bwd without a caller-provided workspace.  The paper
 * has no counterpart: this entry point exists for callers, not for the
 * method.  It is for callers that cannot obtain device scratch memory
 * themselves: a plugin inside a host program whose allocator owns all device
 * memory and offers no way to request scratch, or a latency-critical loop
 * that must not pay cudaMalloc's device-wide synchronisation.  It allocates
 * nothing and calls no allocating routine; the caller still passes every
 * input and output, with the meanings, layouts and errors of rms_bwd.
 *   Scratch: a fixed array of RMS_NOALLOC_SCRATCH_BYTES (32 MiB) inside this
 *   library, held by every device that loads the library until the process
 *   exits.  A shape fits when its workspace need, rms_bwd_workspace_size(M,
 *   N) = min(M, 4 * SMs) * N * 4 bytes rounded up to 256, is at most that:
 *   any M when N <= 32 MiB / (4 * SMs * 4 bytes) (on a 152-SM GB300, N <=
 *   13797; on 148 SMs, N <= 14169), or M * N <= 8388608.  Ask
 *   rms_bwd_workspace_size on the caller's own device; larger shapes are
 *   rejected with RMS_ERR_WORKSPACE before anything else is checked.
 *   M <= 0 or N <= 0 is answered exactly as rms_bwd answers it (M == 0
 *   writes dgamma = 0) without touching the array; every other argument
 *   error is rms_bwd's.
 *   The first call on each device looks up the array's device address with
 *   that device current and caches it; make that first call before any
 *   stream capture.  A device reset (cudaDeviceReset) leaves the cached
 *   address stale: do not use this entry point on a device after resetting
 *   it in the same process.
 *   All calls on a device share the array and it keeps the last call's
 *   contents (nothing in it needs clearing: every partial row the column
 *   sum reads is written earlier in the same call): calls whose executions
 *   overlap on the GPU (other streams, other host threads) race and must be
 *   serialised by the caller.
 */
#define RMS_NOALLOC_SCRATCH_BYTES (32u << 20)
rms_status rms_bwd_noalloc(void* dy, const void* x, const void* gamma, const float* rstd,
                           void* dx, float* dgamma, int64_t M, int64_t N, rms_dtype dtype,
                           int gemma, int inplace_dx, void* stream);

/*
 * rms_fwd_add — residual add fused into the forward: one read of x and of
 * the residual, one write of h and of y, instead of an add kernel whose
 * output is read back by rms_fwd.
 *   h = round(x + residual)   (float32 sum, one rounding to dtype: the
 *                              residual stream keeps the activation type)
 *   y, rstd = rms_fwd(h)      (exactly as rms_fwd on the stored h)
 *   x, residual [M*N] dtype, read; h [M*N] dtype, written (h may be the
 *   residual buffer itself, updating the stream in place; it must not
 *   overlap x, gamma, y or rstd); other arguments as rms_fwd.
 * Source: "02 · 手写 Triton kernel:RMSNorm / RoPE / SwiGLU", sections 1-2
 * (neighbouring elementwise work kept in registers, each tensor read and
 * written once, results written back over an input); the add itself is the
 * residual connection around the normalisation.
 * Errors: as rms_fwd; RMS_ERR_INVALID_ARG when residual or h is NULL.
 */
rms_status rms_fwd_add(const void* x, const void* residual, const void* gamma, void* y, void* h,
                       float* rstd, int64_t M, int64_t N, float eps, rms_dtype dtype, int gemma,
                       void* stream);

/* rms_fwd_add with an explicit row mapping. */
rms_status rms_fwd_add_ex(const void* x, const void* residual, const void* gamma, void* y,
                          void* h, float* rstd, int64_t M, int64_t N, float eps, rms_dtype dtype,
                          int gemma, rms_path path, void* stream);

/*
 * rms_bwd_add — the backward of rms_fwd_add: the gradient reaching h
 * through the residual path is added to the normalisation's input
 * gradient before the one rounding of dx.
 *   dx = round(dRMS(dy; h, gamma, rstd) + dh)   (dRMS as rms_bwd, in float32)
 *   dgamma as rms_bwd (on h).
 *   h [M*N] dtype: the forward's h; dh [M*N] dtype, read; dx [M*N] written,
 *   may be dh itself (accumulating in place) or dy with inplace_dx = 1;
 *   dh must not overlap dy.  Other arguments as rms_bwd.
 * Source: as rms_fwd_add; dRMS as rms_bwd.
 * Errors: as rms_bwd; RMS_ERR_INVALID_ARG when dh is NULL.
 */
rms_status rms_bwd_add(void* dy, const void* h, const void* gamma, const float* rstd,
                       const void* dh, void* dx, float* dgamma, void* workspace, int64_t M,
                       int64_t N, rms_dtype dtype, int gemma, int inplace_dx, void* stream);

/* rms_bwd_add with the workspace size stated and an explicit row mapping. */
rms_status rms_bwd_add_ex(void* dy, const void* h, const void* gamma, const float* rstd,
                          const void* dh, void* dx, float* dgamma, void* workspace,
                          size_t workspace_bytes, int64_t M, int64_t N, rms_dtype dtype,
                          int gemma, int inplace_dx, rms_path path, void* stream);

/*
 * rms_fwd_quant — the forward with its output quantised to FP8 E4M3 in the
 * same pass, for a GEMM that consumes it: y is computed as rms_fwd stores it
 * (same cast order and roundings; r is the same float32 sum of squares,
 * added in the order of the mapping taken, which for rows of more than
 * 2 KiB up to 32 KiB is rms_fwd's own, so there y equals rms_fwd's bit for
 * bit) but never written; instead
 *   amax_i = max_j |y_ij|,  scale_i = amax_i / 448  (1 for an all-zero row)
 *   q_ij   = e4m3(y_ij * (448 / amax_i))   (float32 multiply, then round to
 *            nearest even, saturating at +-448; y_ij ~ e4m3 value * scale_i)
 *   x [M*N] dtype, gamma [N] read; q [M*N] bytes (E4M3: sign, 4 exponent
 *   bits with bias 7, 3 mantissa bits, no infinities), scale [M] and
 *   rstd [M] float32 written; no output may overlap another argument.
 *   Mappings: RMS_PATH_REGISTERS (16-byte aligned rows and pointers, rows
 *   up to 32 KiB), RMS_PATH_CHUNKED (aligned rows of any width: up to 16
 *   slices of 16 KiB, or of 32 KiB for wider rows, a cluster of CTAs per
 *   row reading it once from HBM, the row's sum of squares and maximum |y|
 *   exchanged between them; wider rows a CTA per row, three passes over the
 *   row, the second and third served by L2) or RMS_PATH_SCALAR (any); AUTO
 *   picks the first that fits.
 * Source: y as rms_fwd; the fusion of the consumer's cast as "02 · 手写
 * Triton kernel:RMSNorm / RoPE / SwiGLU", sections 1-2 (neighbouring
 * elementwise work kept in registers, each tensor read or written once).
 * Errors: as rms_fwd; RMS_ERR_UNSUPPORTED for RMS_PATH_STAGED,
 * RMS_ERR_ALIGNMENT for RMS_PATH_REGISTERS / CHUNKED on unaligned rows.
 */
rms_status rms_fwd_quant(const void* x, const void* gamma, uint8_t* q, float* scale, float* rstd,
                         int64_t M, int64_t N, float eps, rms_dtype dtype, int gemma,
                         void* stream);

/* rms_fwd_quant with an explicit row mapping. */
rms_status rms_fwd_quant_ex(const void* x, const void* gamma, uint8_t* q, float* scale,
                            float* rstd, int64_t M, int64_t N, float eps, rms_dtype dtype,
                            int gemma, rms_path path, void* stream);

/*
 * ln_fwd — forward LayerNorm over M rows of N, on the same engine.
 *   mean_i = (1/N) sum_j x_ij,  var_i = (1/N) sum_j (x_ij - mean_i)^2,
 *   rstd_i = 1/sqrt(var_i + eps),  y_ij = (x_ij - mean_i) * rstd_i * w_j + b_j
 *   x [M*N], w [N], b [N] (or NULL: no bias), y [M*N]; mean, rstd [M] float32,
 *   written for ln_bwd.  Types as rms_dtype (w and b share the weight type).
 *   Arithmetic float32, the variance from the centred values (two passes
 *   over the row held on chip), one rounding per stored y.
 * Source: "第 07 章:LayerNorm——反向传播与原子锁", step 3 (forward kernel).
 * Errors: RMS_ERR_INVALID_ARG, RMS_ERR_UNSUPPORTED, RMS_ERR_CUDA.
 */
rms_status ln_fwd(const void* x, const void* w, const void* b, void* y, float* mean, float* rstd,
                  int64_t M, int64_t N, float eps, rms_dtype dtype, void* stream);

/* ln_fwd with an explicit mapping (RMS_PATH_REGISTERS or RMS_PATH_SCALAR). */
rms_status ln_fwd_ex(const void* x, const void* w, const void* b, void* y, float* mean,
                     float* rstd, int64_t M, int64_t N, float eps, rms_dtype dtype, rms_path path,
                     void* stream);

/*
 * ln_bwd — backward LayerNorm from the saved mean and rstd.
 *   xhat = (x - mean)*rstd, g = dy*w, c1 = mean_j(xhat*g), c2 = mean_j(g),
 *   dx = (g - (xhat*c1 + c2)) * rstd,
 *   dw_j = sum_i dy_ij*xhat_ij,  db_j = sum_i dy_ij   (sums over rows)
 *   dy, x [M*N]; w [N]; mean, rstd [M] float32; dx [M*N] (NULL or dy with
 *   inplace_dx = 1); dw [N] float32; db [N] float32 or NULL (not computed);
 *   workspace of ln_bwd_workspace_size(M, N) bytes, 256-byte aligned.
 * dw and db come from per-CTA partials over a static row assignment and a
 * fixed-order column sum (no atomics, no locks): bitwise reproducible.
 * Source: "第 07 章:LayerNorm——反向传播与原子锁", § 3.0 (backward formulas,
 * row contributions summed over rows).
 * Errors: as rms_bwd.
 */
rms_status ln_bwd(void* dy, const void* x, const void* w, const float* mean, const float* rstd,
                  void* dx, float* dw, float* db, void* workspace, int64_t M, int64_t N,
                  rms_dtype dtype, int inplace_dx, void* stream);

/* ln_bwd with the workspace size stated and an explicit mapping
 * (RMS_PATH_STAGED or RMS_PATH_SCALAR). */
rms_status ln_bwd_ex(void* dy, const void* x, const void* w, const float* mean,
                     const float* rstd, void* dx, float* dw, float* db, void* workspace,
                     size_t workspace_bytes, int64_t M, int64_t N, rms_dtype dtype, int inplace_dx,
                     rms_path path, void* stream);

/* ln_bwd_reduction — as rms_bwd_reduction, for ln_bwd's dw and db (each is
 * summed through P partial rows of at most rows_per_partial rows; path
 * RMS_PATH_AUTO, RMS_PATH_STAGED or RMS_PATH_SCALAR).
 * Source: "第 07 章:LayerNorm——反向传播与原子锁", § 3.0 (row contributions
 * summed over rows). */
rms_status ln_bwd_reduction(int64_t M, int64_t N, rms_dtype dtype, rms_path path,
                            int64_t* partials, int64_t* rows_per_partial);

/* Bytes of workspace ln_bwd needs for M rows of N on the current device
 * (two rows of partials per CTA: dw and db; a multiple of 256). */
size_t ln_bwd_workspace_size(int64_t M, int64_t N);

/* Bytes of workspace rms_bwd needs for M rows of N on the current device
 * (an upper bound over dtypes and mappings, a multiple of 256).  Returns 0
 * for M <= 0 or N <= 0, and 0 if the device cannot be queried. */
size_t rms_bwd_workspace_size(int64_t M, int64_t N);

/* Static, NUL-terminated description of a status code. */
const char* rms_status_string(rms_status status);

/* Synchronises `stream`, then reports and clears the device-side status
 * words of the current device: RMS_ERR_TIMEOUT if a bounded wait in a
 * staged mapping (RMSNorm or LayerNorm) gave up since the last query (that launch's outputs are
 * then incomplete), RMS_ERR_CUDA if the stream reports an error, else
 * RMS_OK. */
rms_status rms_last_device_status(void* stream);

/* Poll limit of the staged mapping's mbarrier waits, for all later launches
 * in this process; returns the previous value.  A negative value restores
 * the default.  A limit of 0 makes every wait give up at once, which lets a
 * test exercise the timeout path without hanging anything. */
int64_t rms_set_wait_limit(int64_t polls);

/* Number of kernels the library launched since the process started (all
 * devices), for accounting in benchmarks. */
uint64_t rms_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_H_ */
