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

// The same sum for N % 4 == 0 with 16-byte loads.  A CTA of 512 threads
// covers L float4 columns with S = 512 / L row strands (L a power of two,
// chosen on the host from P and N).  Strand t sums rows t, t+S, t+2S, ... in
// increasing order, eight rows loaded before any is added so that a strand's
// loads are in flight together; the S strand sums are then combined by a
// fixed radix-8 tree (strand t adds t+h, t+2h, ... in order at each level).
// blockIdx.y picks one of two (ws, out) pairs so that two column sums
// (LayerNorm's dw and db) share one launch.  The order depends only on P and
// N, so the sums are reproducible bit for bit.
__global__ void __launch_bounds__(512)
rms_colreduce4_kernel(const float4* __restrict__ ws0, float4* __restrict__ out0,
                      const float4* __restrict__ ws1, float4* __restrict__ out1, int64_t P,
                      int N4, int log2L) {
  __shared__ float4 part[512];
  const int L = 1 << log2L;
  const int S = 512 >> log2L;
  const int cx = threadIdx.x & (L - 1);
  const int strand = threadIdx.x >> log2L;
  const float4* ws = blockIdx.y ? ws1 : ws0;
  float4* out = blockIdx.y ? out1 : out0;
  const int64_t col4 = (int64_t)blockIdx.x * L + cx;
  pdl_wait();
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col4 < N4) {
    const float4* src = ws + col4;
    for (int64_t p0 = strand; p0 < P; p0 += 8 * (int64_t)S) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t p = p0 + (int64_t)u * S;
        if (p < P) v[u] = src[p * N4];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (p0 + (int64_t)u * S < P) {
          s.x += v[u].x; s.y += v[u].y; s.z += v[u].z; s.w += v[u].w;
        }
      }
    }
  }
  part[threadIdx.x] = s;
  for (int h = S; h > 1;) {
    const int g = h >= 8 ? 8 : h;
    const int hn = h / g;
    __syncthreads();
    if (strand < hn) {
      float4 t = part[threadIdx.x];
      for (int q = 1; q < g; ++q) {
        const float4 u = part[((strand + q * hn) << log2L) + cx];
        t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
      }
      part[threadIdx.x] = t;
    }
    h = hn;
  }
  if (strand == 0 && col4 < N4) {
    if (S > 1) s = part[cx];
    out[col4] = s;
  }
}

// out[j] = parts[0][j] + parts[1][j] + ... + parts[R-1][j], added one row
// at a time in increasing row order (one float32 rounding per addition).
// The rows are the per-rank dgamma vectors of a row-sharded backward, so the
// total is the same on every rank and does not depend on how they were
// exchanged.  A thread owns four columns (one float4 when aligned).
__global__ void __launch_bounds__(256)
rms_rank_sum_kernel(const float* __restrict__ parts, float* __restrict__ out, int64_t R, int64_t N,
                    int vec) {
  pdl_wait();
  const int64_t j0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (j0 >= N) return;
  if (vec) {  // N % 4 == 0 and both pointers 16-byte aligned
    const float4* p4 = reinterpret_cast<const float4*>(parts) + j0 / 4;
    float4 s = p4[0];
    for (int64_t r = 1; r < R; ++r) {
      const float4 v = p4[r * (N / 4)];
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    reinterpret_cast<float4*>(out)[j0 / 4] = s;
    return;
  }
  for (int64_t j = j0; j < j0 + 4 && j < N; ++j) {
    float s = parts[j];
    for (int64_t r = 1; r < R; ++r) s += parts[r * N + j];
    out[j] = s;
  }
}


// dst[j] = src[j] rounded to the weight type W (round to nearest even; a
// copy for float32): the float32 column sum handed back in the weight's own
// type.  Four columns per thread, 16-byte loads when aligned.
template <typename W>
__global__ void __launch_bounds__(256)
rms_weight_cast_kernel(const float* __restrict__ src, W* __restrict__ dst, int64_t N, int vec) {
  pdl_wait();
  const int64_t j0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (j0 >= N) return;
  if (vec) {  // N % 4 == 0, src 16-byte and dst 4 * sizeof(W)-byte aligned
    const float4 v = reinterpret_cast<const float4*>(src)[j0 / 4];
    if constexpr (sizeof(W) == 4) {
      reinterpret_cast<float4*>(dst)[j0 / 4] = v;
    } else {
      const uint2 o = make_uint2(Half2Ops<W>::narrow(pk2(v.x, v.y)),
                                 Half2Ops<W>::narrow(pk2(v.z, v.w)));
      reinterpret_cast<uint2*>(dst)[j0 / 4] = o;
    }
    return;
  }
  for (int64_t j = j0; j < j0 + 4 && j < N; ++j) dst[j] = Elem<W>::from_f(src[j]);
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

// Lanes per CTA for the vectorised column sum: at most eight rows per strand,
// then narrower slabs (more CTAs) until the grid has a CTA per SM.  (A grid
// past one resident wave, or a dependent launch triggered early, measured
// slower on GB300: the column sum sits between two row kernels.)
static int colreduce_log2_lanes(int64_t P, int N4, int sms) {
  int log2S = 0;
  while (log2S < 8 && ((int64_t)8 << log2S) < P) ++log2S;
  while (log2S < 8 && ((int64_t)N4 >> (9 - log2S)) < (int64_t)sms) ++log2S;
  return 9 - log2S;
}

cudaError_t launch_colreduce2(const float* ws0, float* out0, const float* ws1, float* out1,
                              int64_t P, int N, int sms, cudaStream_t s) {
  const bool two = ws1 != nullptr;
  const bool vec = N % 4 == 0 && !((uintptr_t)ws0 & 15u) && !((uintptr_t)out0 & 15u) &&
                   (!two || (!((uintptr_t)ws1 & 15u) && !((uintptr_t)out1 & 15u)));
  if (!vec) {
    cudaError_t e = rmsk::launch_pdl(rmsk::rms_dgamma_colreduce_kernel,
                                     dim3((unsigned)((N + 31) / 32)), dim3(256), 0, s, ws0, out0,
                                     P, N);
    if (e != cudaSuccess || !two) return e;
    return rmsk::launch_pdl(rmsk::rms_dgamma_colreduce_kernel, dim3((unsigned)((N + 31) / 32)),
                            dim3(256), 0, s, ws1, out1, P, N);
  }
  const int N4 = N / 4;
  const int log2L = colreduce_log2_lanes(P, N4, sms);
  const int L = 1 << log2L;
  return rmsk::launch_pdl(rmsk::rms_colreduce4_kernel,
                          dim3((unsigned)((N4 + L - 1) / L), two ? 2u : 1u), dim3(512), 0, s,
                          reinterpret_cast<const float4*>(ws0), reinterpret_cast<float4*>(out0),
                          reinterpret_cast<const float4*>(two ? ws1 : ws0),
                          reinterpret_cast<float4*>(two ? out1 : out0), P, N4, log2L);
}

cudaError_t launch_colreduce(const float* ws, float* dgamma, int64_t P, int N, int sms,
                             cudaStream_t s) {
  return launch_colreduce2(ws, dgamma, nullptr, nullptr, P, N, sms, s);
}

cudaError_t launch_rank_sum(const float* parts, float* out, int64_t R, int64_t N,
                            cudaStream_t s) {
  const int vec = N % 4 == 0 && !((uintptr_t)parts & 15u) && !((uintptr_t)out & 15u);
  const int64_t threads = (N + 3) / 4;
  return rmsk::launch_pdl(rmsk::rms_rank_sum_kernel, dim3((unsigned)((threads + 255) / 256)),
                          dim3(256), 0, s, parts, out, R, N, vec);
}

cudaError_t launch_weight_cast(const float* src, void* dst, int64_t N, int dtype,
                               cudaStream_t s) {
  const int wb = weight_bytes(dtype);
  const int vec = N % 4 == 0 && !((uintptr_t)src & 15u) && !((uintptr_t)dst & (4u * wb - 1u));
  const int64_t threads = (N + 3) / 4;
  const dim3 grid((unsigned)((threads + 255) / 256)), block(256);
  switch (dtype) {
    case kBF16:
      return rmsk::launch_pdl(rmsk::rms_weight_cast_kernel<__nv_bfloat16>, grid, block, 0, s, src,
                              static_cast<__nv_bfloat16*>(dst), N, vec);
    case kF16:
      return rmsk::launch_pdl(rmsk::rms_weight_cast_kernel<__half>, grid, block, 0, s, src,
                              static_cast<__half*>(dst), N, vec);
    default:
      return rmsk::launch_pdl(rmsk::rms_weight_cast_kernel<float>, grid, block, 0, s, src,
                              static_cast<float*>(dst), N, vec);
  }
}

}  // namespace rmsi
