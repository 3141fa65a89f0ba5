// Scalar-load RMSNorm kernels for rows that are not 16-byte aligned (odd N,
// offset pointers), and the column reduction that finishes dgamma for every
// backward mapping.
//
// The scalar kernels compute exactly what the vector kernels compute (same
// formulas, same cast order, float32 accumulation) but read elements one at
// a time with a CTA per row, touching x twice (the second read is served by
// L1/L2).  The backward keeps its dgamma column partials in shared memory,
// one slot per column owned by one thread, and is persistent with a static
// row assignment like the register mapping.
//
// Sources: "Hướng dẫn Triton RMSNorm: kernel, backward…", sections "Vấn đề
// và công thức tham chiếu", "Vì sao cần một lượt đi và một lượt về?",
// "Reduce dgamma không có race khi ghi" (second pass summing the partials
// column by column), "Tổng không phải trung bình".
#include "common.cuh"
#include "internal.h"

namespace rmsk {

constexpr int kScalarThreads = 256;

template <typename T, typename W>
__global__ void __launch_bounds__(kScalarThreads)
rms_fwd_scalar_kernel(const T* __restrict__ x, const W* __restrict__ gamma, T* __restrict__ y,
                      float* __restrict__ rstd, int64_t M, int N, float eps, int gemma,
                      const T* res, T* h) {
  using E = Elem<T>;
  __shared__ float red[kScalarThreads / 32];
  const int64_t row = blockIdx.x;
  const T* xr = x + row * N;
  pdl_trigger();
  pdl_wait();
  Kahan1 acc;  // a thread adds N / kScalarThreads squares in sequence
  for (int j = threadIdx.x; j < N; j += kScalarThreads) {
    float f = E::to_f(xr[j]);
    if (res) {  // fused residual add: h = x + res, rounded to T, stored and normalised
      const T hv = E::from_f(f + E::to_f(res[row * N + j]));
      h[row * N + j] = hv;
      f = E::to_f(hv);
    }
    acc.add(__fmul_rn(f, f));
  }
  if (res) xr = h + row * N;  // the second pass reads h back (this thread's own elements)
  const float ss = group_sum(acc.total(), kScalarThreads, 0, red);
  const float r = 1.0f / sqrtf(ss / (float)N + eps);
  if (threadIdx.x == 0) rstd[row] = r;
  T* yr = y + row * N;
  for (int j = threadIdx.x; j < N; j += kScalarThreads) {
    const float f = E::to_f(xr[j]);
    const float g = Elem<W>::to_f(gamma[j]);
    const float o = gemma ? (f * r) * (1.0f + g) : Elem<W>::round(f * r) * g;
    yr[j] = E::from_f(o);
  }
}

template <typename T, typename W>
__global__ void __launch_bounds__(kScalarThreads)
rms_bwd_scalar_kernel(const T* dy, const T* __restrict__ x, const W* __restrict__ gamma,
                      const float* __restrict__ rstd, T* dx, float* __restrict__ ws, int64_t M,
                      int N, int gemma, int acc_in_smem, const T* dh) {
  using E = Elem<T>;
  __shared__ float red[2][kScalarThreads / 32];
  // dgamma partials of this CTA, column j owned by thread j % kScalarThreads:
  // in shared memory when N floats fit, else in the CTA's workspace row.
  extern __shared__ float acc_s[];
  float* acc = acc_in_smem ? acc_s : ws + (int64_t)blockIdx.x * N;
  pdl_wait();
  for (int j = threadIdx.x; j < N; j += kScalarThreads) acc[j] = 0.f;

  int it = 0;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x, ++it) {
    const T* xr = x + row * N;
    const T* dr = dy + row * N;
    const float r = rstd[row];
    // xn = x*r, u = dy*w:  k = mean(u*xn) = r*c,  dx = r*(u - xn*k).
    Kahan1 dot;
    for (int j = threadIdx.x; j < N; j += kScalarThreads) {
      const float g = Elem<W>::to_f(gamma[j]);
      const float w = gemma ? 1.0f + g : g;
      dot.add(__fmul_rn(E::to_f(dr[j]) * w, E::to_f(xr[j]) * r));
    }
    const float s = group_sum(dot.total(), kScalarThreads, 0, red[it & 1]);
    const float k = s / (float)N;
    T* out = dx + row * N;
    for (int j = threadIdx.x; j < N; j += kScalarThreads) {
      const float xn = E::to_f(xr[j]) * r;
      const float d = E::to_f(dr[j]);
      const float g = Elem<W>::to_f(gamma[j]);
      const float w = gemma ? 1.0f + g : g;
      acc[j] = fmaf(d, xn, acc[j]);
      const float o = fmaf(-xn, k, d * w) * r;
      out[j] = E::from_f(dh ? o + E::to_f(dh[row * N + j]) : o);  // fused residual gradient
    }
  }
  if (acc_in_smem) {
    float* wp = ws + (int64_t)blockIdx.x * N;
    for (int j = threadIdx.x; j < N; j += kScalarThreads) wp[j] = acc[j];
  }
}

// dgamma[j] = sum over p = 0..P-1 of ws[p][j].  A CTA covers 32 columns with
// 8 row-strands: strand t sums rows t, t+8, t+16, ... in increasing order,
// then strand sums are added in strand order.  Fixed order, no atomics.
__global__ void __launch_bounds__(256)
rms_dgamma_colreduce_kernel(const float* __restrict__ ws, float* __restrict__ dgamma, int64_t P,
                            int N) {
  __shared__ float part[8][33];
  const int tx = threadIdx.x & 31;
  const int ty = threadIdx.x >> 5;
  const int64_t col = (int64_t)blockIdx.x * 32 + tx;
  pdl_wait();
  float s = 0.f;
  if (col < N) {
    for (int64_t p = ty; p < P; p += 8) s += ws[p * N + col];
  }
  part[ty][tx] = s;
  __syncthreads();
  if (ty == 0 && col < N) {
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) t += part[q][tx];
    dgamma[col] = t;
  }
}

// The same sum for N % 4 == 0 with 16-byte loads: a CTA covers 32 columns
// (8 float4 lanes) with 32 row strands; strand t sums rows t, t+32, ... in
// increasing order with four independent float4 loads in flight, then the 32
// strand sums are added in strand order.
__global__ void __launch_bounds__(256)
rms_dgamma_colreduce4_kernel(const float4* __restrict__ ws, float4* __restrict__ dgamma,
                             int64_t P, int N4) {
  __shared__ float4 part[32][9];
  const int cx = threadIdx.x & 7;
  const int strand = threadIdx.x >> 3;
  const int64_t col4 = (int64_t)blockIdx.x * 8 + cx;
  pdl_wait();
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col4 < N4) {
    const float4* src = ws + col4;
    int64_t p = strand;
    for (; p + 96 < P; p += 128) {
      const float4 a = src[p * N4], b = src[(p + 32) * N4], c = src[(p + 64) * N4],
                   d = src[(p + 96) * N4];
      s.x += a.x; s.y += a.y; s.z += a.z; s.w += a.w;
      s.x += b.x; s.y += b.y; s.z += b.z; s.w += b.w;
      s.x += c.x; s.y += c.y; s.z += c.z; s.w += c.w;
      s.x += d.x; s.y += d.y; s.z += d.z; s.w += d.w;
    }
    for (; p < P; p += 32) {
      const float4 a = src[p * N4];
      s.x += a.x; s.y += a.y; s.z += a.z; s.w += a.w;
    }
  }
  part[strand][cx] = s;
  __syncthreads();
  if (strand == 0 && col4 < N4) {
    float4 t = part[0][cx];
    for (int q = 1; q < 32; ++q) {
      const float4 u = part[q][cx];
      t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
    }
    dgamma[col4] = t;
  }
}

}  // namespace rmsk

namespace rmsi {

bool plan_scalar(int N, int dtype, bool bwd, const DeviceInfo& d, Mapping* m) {
  (void)dtype;
  if (N <= 0) return false;
  m->path = kScalar;
  m->G = rmsk::kScalarThreads;
  m->kv = 0;
  m->threads = rmsk::kScalarThreads;
  m->rows_per_cta = 1;
  m->smem = bwd ? (size_t)N * sizeof(float) : 0;
  m->smem_acc = 1;
  if (m->smem + 1024 > d.smem_optin) {  // room for the static reduction slots
    m->smem = 0;                         // too wide: partials in the workspace rows
    m->smem_acc = 0;
  }
  return true;
}

template <typename T, typename W>
static cudaError_t launch_fwd_scalar_t(const FwdArgs& a, dim3 grid, dim3 block, cudaStream_t s) {
  return rmsk::launch_pdl(rmsk::rms_fwd_scalar_kernel<T, W>, grid, block, 0, s,
                          static_cast<const T*>(a.x), static_cast<const W*>(a.gamma),
                          static_cast<T*>(a.y), a.rstd, a.M, a.N, a.eps, a.gemma,
                          static_cast<const T*>(a.res), static_cast<T*>(a.h));
}

cudaError_t launch_fwd_scalar(const FwdArgs& a, const Mapping& m, cudaStream_t s) {
  const dim3 grid((unsigned)a.M), block(m.threads);
  switch (a.dtype) {
    case kBF16: return launch_fwd_scalar_t<__nv_bfloat16, __nv_bfloat16>(a, grid, block, s);
    case kF16: return launch_fwd_scalar_t<__half, __half>(a, grid, block, s);
    case kBF16W32: return launch_fwd_scalar_t<__nv_bfloat16, float>(a, grid, block, s);
    case kF16W32: return launch_fwd_scalar_t<__half, float>(a, grid, block, s);
    default: return launch_fwd_scalar_t<float, float>(a, grid, block, s);
  }
}

template <typename T, typename W>
static const void* bwd_scalar_ptr() {
  return reinterpret_cast<const void*>(&rmsk::rms_bwd_scalar_kernel<T, W>);
}

cudaError_t size_bwd_scalar(const BwdArgs& a, const DeviceInfo& d, Mapping* m) {
  const void* k;
  switch (a.dtype) {
    case kBF16: k = bwd_scalar_ptr<__nv_bfloat16, __nv_bfloat16>(); break;
    case kF16: k = bwd_scalar_ptr<__half, __half>(); break;
    case kBF16W32: k = bwd_scalar_ptr<__nv_bfloat16, float>(); break;
    case kF16W32: k = bwd_scalar_ptr<__half, float>(); break;
    default: k = bwd_scalar_ptr<float, float>(); break;
  }
  cudaError_t e = opt_in_max_smem(k, d);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, m->threads, m->smem);
  if (e != cudaSuccess) return e;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  int64_t P = (int64_t)occ * d.sms;
  if (P > max_partials(d.sms)) P = max_partials(d.sms);
  if (P > a.M) P = a.M;
  if (P < 1) P = 1;
  m->blocks = P;
  m->partials = P;
  return cudaSuccess;
}

template <typename T, typename W>
static cudaError_t launch_bwd_scalar_t(const BwdArgs& a, const Mapping& m, cudaStream_t s) {
  const dim3 grid((unsigned)m.blocks), block(m.threads);
  return rmsk::launch_pdl(rmsk::rms_bwd_scalar_kernel<T, W>, grid, block, m.smem, s,
                          static_cast<const T*>(a.dy), static_cast<const T*>(a.x),
                          static_cast<const W*>(a.gamma), a.rstd, static_cast<T*>(a.dx), a.ws,
                          a.M, a.N, a.gemma, m.smem_acc, static_cast<const T*>(a.dh));
}

cudaError_t launch_bwd_scalar(const BwdArgs& a, const Mapping& m, cudaStream_t s) {
  switch (a.dtype) {
    case kBF16: return launch_bwd_scalar_t<__nv_bfloat16, __nv_bfloat16>(a, m, s);
    case kF16: return launch_bwd_scalar_t<__half, __half>(a, m, s);
    case kBF16W32: return launch_bwd_scalar_t<__nv_bfloat16, float>(a, m, s);
    case kF16W32: return launch_bwd_scalar_t<__half, float>(a, m, s);
    default: return launch_bwd_scalar_t<float, float>(a, m, s);
  }
}

cudaError_t launch_colreduce(const float* ws, float* dgamma, int64_t P, int N, cudaStream_t s) {
  if (N % 4 != 0 || ((uintptr_t)ws & 15u) || ((uintptr_t)dgamma & 15u))
    return rmsk::launch_pdl(rmsk::rms_dgamma_colreduce_kernel, dim3((unsigned)((N + 31) / 32)),
                            dim3(256), 0, s, ws, dgamma, P, N);
  const int N4 = N / 4;
  return rmsk::launch_pdl(rmsk::rms_dgamma_colreduce4_kernel, dim3((unsigned)((N4 + 7) / 8)),
                          dim3(256), 0, s, reinterpret_cast<const float4*>(ws),
                          reinterpret_cast<float4*>(dgamma), P, N4);
}

}  // namespace rmsi
