// RMSNorm for rows of any width: the row is never held on chip, so every
// pass streams it from memory.  Forward: a row pass computes r (into rstd),
// then a normalise pass over (row, chunk) units writes y.  Backward: a row
// pass computes k = r * mean(u * x) per row, then (row group, chunk) units
// write dx and keep dgamma partials for their chunk's columns in registers
// across the group's rows; the fixed-order column reduction finishes dgamma.
// Three passes over x (and dy) instead of two, no shared-memory limit on N.
//
// Sources: "Hướng dẫn Triton RMSNorm: kernel, backward…", sections "Vấn đề
// và công thức tham chiếu" (r, y) and "Backward đầu vào: giữ đúng N" (dx,
// dgamma); the looped row reduction for rows wider than one block is the
// LN chapter's ("第 07 章:LayerNorm——反向传播与原子锁", step 3).
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace rmsk {

constexpr int kChunkThreads = 512;
constexpr int kChunkVecs = 4;                             // 16-byte vectors per thread per chunk
constexpr int kChunkSpan = kChunkThreads * kChunkVecs;    // vectors per chunk

// Sum over the CTA; `red` is [2][kChunkThreads / 32], alternated by `buf`
// so that consecutive calls need one barrier each.
__device__ __forceinline__ float cta_sum(float v, float* red, int buf) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31;
  if (lane == 0) red[buf * 32 + (threadIdx.x >> 5)] = v;
  __syncthreads();
  return warp_sum(lane < kChunkThreads / 32 ? red[buf * 32 + lane] : 0.f);
}

// One CTA per row at a time (grid-stride over rows).  Forward: out = r =
// 1/sqrt(sum(x^2)/N + eps); with RES the row is h = x + res, stored to h for
// the normalise pass.  Backward: out = k = sum(u * x * r)/N.
template <typename T, typename W, bool GEMMA, bool BWD, bool RES>
__global__ void __launch_bounds__(kChunkThreads)
rms_rowstat_kernel(const T* __restrict__ x, const T* __restrict__ dy, const W* __restrict__ gamma,
                   const float* __restrict__ rstd_in, float* __restrict__ out, int64_t M, int N,
                   float eps, const T* res, T* h) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  __shared__ float red[2 * 32];
  const int NV = N / VN;
  pdl_wait();
  int buf = 0;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x, buf ^= 1) {
    const uint4* xr = reinterpret_cast<const uint4*>(x) + row * (int64_t)NV;
    const uint4* dr = reinterpret_cast<const uint4*>(dy) + row * (int64_t)NV;
    const float r = BWD ? rstd_in[row] : 0.f;
    Kahan2 acc;  // a thread adds NV / kChunkSpan partial sums in sequence
    for (int v0 = threadIdx.x; v0 < NV; v0 += kChunkSpan) {
      uint4 xv[kChunkVecs], dv[kChunkVecs];
#pragma unroll
      for (int u = 0; u < kChunkVecs; ++u) {
        const int v = v0 + u * kChunkThreads;
        xv[u] = v < NV ? ld_keep(xr + v) : make_uint4(0u, 0u, 0u, 0u);
        if (BWD || RES) {
          const uint4* src = BWD ? dr : reinterpret_cast<const uint4*>(res) + row * (int64_t)NV;
          dv[u] = v < NV ? ld_stream(src + v) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (RES) {
#pragma unroll
        for (int u = 0; u < kChunkVecs; ++u) {
          const int v = v0 + u * kChunkThreads;
          xv[u] = Math::add_round(xv[u], dv[u]);
          if (v < NV) __stcg(reinterpret_cast<uint4*>(h) + row * (int64_t)NV + v, xv[u]);
        }
      }
      f32x2 part = 0ull;
#pragma unroll
      for (int u = 0; u < kChunkVecs; ++u) {
        const int v = v0 + u * kChunkThreads;
        if (v < NV) {
          if (BWD) {
            Math::backward_dot(xv[u], dv[u], GV::load(gamma, v), r, part);
          } else {
            Math::sumsq(xv[u], part);
          }
        }
      }
      acc.add(part);
    }
    const float tot = cta_sum(acc.total(), red, buf);
    if (threadIdx.x == 0) out[row] = BWD ? tot / (float)N : 1.0f / sqrtf(tot / (float)N + eps);
  }
}

// y over (row, chunk) units, grid-stride.
template <typename T, typename W, bool GEMMA>
__global__ void __launch_bounds__(kChunkThreads)
rms_fwd_chunk_kernel(const T* __restrict__ x, const W* __restrict__ gamma, T* __restrict__ y,
                     const float* __restrict__ rstd, int64_t M, int N, int nchunks) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  const int NV = N / VN;
  pdl_wait();
  const int64_t units = M * (int64_t)nchunks;
  for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int64_t row = unit / nchunks;
    const int c = (int)(unit - row * nchunks);
    const float r = rstd[row];
    const uint4* xr = reinterpret_cast<const uint4*>(x) + row * (int64_t)NV;
    uint4* yr = reinterpret_cast<uint4*>(y) + row * (int64_t)NV;
    const int v0 = c * kChunkSpan + threadIdx.x;
    uint4 xv[kChunkVecs];
#pragma unroll
    for (int u = 0; u < kChunkVecs; ++u) {
      const int v = v0 + u * kChunkThreads;
      xv[u] = v < NV ? ld_stream(xr + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kChunkVecs; ++u) {
      const int v = v0 + u * kChunkThreads;
      if (v < NV) st_stream(yr + v, Math::forward(xv[u], GV::load(gamma, v), r));
    }
  }
}

// dx over (row group, chunk) units: unit = (rg, c) takes rows rg, rg + RG,
// ... in increasing order, and writes its dgamma partial for chunk c's
// columns into workspace row rg.
template <typename T, typename W, bool GEMMA, bool RES>
__global__ void __launch_bounds__(kChunkThreads)
rms_bwd_chunk_kernel(const T* dy, const T* __restrict__ x, const W* __restrict__ gamma,
                     const float* __restrict__ rstd, const float* __restrict__ kbuf, T* dx,
                     float* __restrict__ ws, int64_t M, int N, int nchunks, int64_t RG,
                     const T* dh) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  constexpr int NP = Math::kPairs;
  const int NV = N / VN;
  pdl_wait();
  const int64_t rg = blockIdx.x / nchunks;
  const int c = (int)(blockIdx.x - rg * nchunks);
  const int v0 = c * kChunkSpan + threadIdx.x;
  GV gv[kChunkVecs];
  f32x2 acc[kChunkVecs][NP];
#pragma unroll
  for (int u = 0; u < kChunkVecs; ++u) {
    const int v = v0 + u * kChunkThreads;
    gv[u] = v < NV ? GV::load(gamma, v) : GV::zero();
#pragma unroll
    for (int e = 0; e < NP; ++e) acc[u][e] = 0ull;
  }
  for (int64_t row = rg; row < M; row += RG) {
    const float r = rstd[row];
    const float k = kbuf[row];
    const uint4* xr = reinterpret_cast<const uint4*>(x) + row * (int64_t)NV;
    const uint4* dr = reinterpret_cast<const uint4*>(dy) + row * (int64_t)NV;
    uint4* out = reinterpret_cast<uint4*>(dx) + row * (int64_t)NV;
    uint4 xv[kChunkVecs], dv[kChunkVecs];
#pragma unroll
    for (int u = 0; u < kChunkVecs; ++u) {
      const int v = v0 + u * kChunkThreads;
      const bool in = v < NV;
      xv[u] = in ? ld_stream(xr + v) : make_uint4(0u, 0u, 0u, 0u);
      dv[u] = in ? ld_stream(dr + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kChunkVecs; ++u) {
      const int v = v0 + u * kChunkThreads;
      if (v < NV) {
        Math::backward_acc(xv[u], dv[u], r, acc[u]);
        const uint4 hv = RES ? ld_stream(reinterpret_cast<const uint4*>(dh) + row * (int64_t)NV + v)
                             : make_uint4(0u, 0u, 0u, 0u);
        st_stream(out + v, RES ? Math::backward_dx_add(xv[u], dv[u], gv[u], r, k, hv)
                               : Math::backward_dx(xv[u], dv[u], gv[u], r, k));
      }
    }
  }
  float* wp = ws + rg * (int64_t)N;
#pragma unroll
  for (int u = 0; u < kChunkVecs; ++u) {
    const int v = v0 + u * kChunkThreads;
    if (v < NV) {
      float4* w4 = reinterpret_cast<float4*>(wp + (int64_t)v * VN);
#pragma unroll
      for (int q = 0; q < NP / 2; ++q)
        w4[q] = make_float4(lo2(acc[u][2 * q]), hi2(acc[u][2 * q]), lo2(acc[u][2 * q + 1]),
                            hi2(acc[u][2 * q + 1]));
    }
  }
}

template <typename F>
cudaError_t with_types(int dtype, int gemma, bool res, F&& f) {
  auto g = [&](auto* tp, auto* wp) -> cudaError_t {
    if (res) return gemma ? f(tp, wp, std::true_type{}, std::true_type{})
                          : f(tp, wp, std::false_type{}, std::true_type{});
    return gemma ? f(tp, wp, std::true_type{}, std::false_type{})
                 : f(tp, wp, std::false_type{}, std::false_type{});
  };
  switch (dtype) {
    case rmsi::kBF16: return g((__nv_bfloat16*)nullptr, (__nv_bfloat16*)nullptr);
    case rmsi::kF16: return g((__half*)nullptr, (__half*)nullptr);
    case rmsi::kBF16W32: return g((__nv_bfloat16*)nullptr, (float*)nullptr);
    case rmsi::kF16W32: return g((__half*)nullptr, (float*)nullptr);
    default: return g((float*)nullptr, (float*)nullptr);
  }
}

}  // namespace rmsk

namespace rmsi {

bool plan_chunked(int N, int dtype, Mapping* m) {
  const int64_t row_bytes = (int64_t)N * dtype_bytes(dtype);
  if (N <= 0 || row_bytes % 16 != 0) return false;
  const int64_t NV = row_bytes / 16;
  m->path = kChunked;
  m->cluster = 1;
  m->threads = rmsk::kChunkThreads;
  m->kv = rmsk::kChunkVecs;
  m->G = rmsk::kChunkThreads;
  m->rows_per_cta = 1;
  m->chunks = (int)((NV + rmsk::kChunkSpan - 1) / rmsk::kChunkSpan);
  m->smem = 0;
  return true;
}

cudaError_t launch_fwd_chunked(const FwdArgs& a, const Mapping& m, const DeviceInfo& d,
                               cudaStream_t s) {
  return rmsk::with_types(a.dtype, a.gemma, a.res != nullptr,
                         [&](auto* tp, auto* wp, auto gm, auto rs) -> cudaError_t {
    using T = std::remove_pointer_t<decltype(tp)>;
    using W = std::remove_pointer_t<decltype(wp)>;
    constexpr bool GEMMA = decltype(gm)::value;
    constexpr bool RES = decltype(rs)::value;
    const T* x = static_cast<const T*>(a.x);
    const W* g = static_cast<const W*>(a.gamma);
    const int64_t rows_grid = std::min<int64_t>(a.M, (int64_t)d.sms * 4);
    cudaError_t e = rmsk::launch_pdl(rmsk::rms_rowstat_kernel<T, W, GEMMA, false, RES>,
                               dim3((unsigned)rows_grid), dim3(rmsk::kChunkThreads), 0, s, x,
                               (const T*)nullptr, g, (const float*)nullptr, a.rstd, a.M, a.N,
                               a.eps, static_cast<const T*>(a.res), static_cast<T*>(a.h));
    if (e != cudaSuccess) return e;
    const int64_t units = a.M * (int64_t)m.chunks;
    const int64_t grid = std::min<int64_t>(units, (int64_t)d.sms * 16);
    // With a residual the normalise pass reads h, which the row pass wrote.
    const T* src = RES ? static_cast<const T*>(a.h) : x;
    return rmsk::launch_pdl(rmsk::rms_fwd_chunk_kernel<T, W, GEMMA>, dim3((unsigned)grid),
                      dim3(rmsk::kChunkThreads), 0, s, src, g, static_cast<T*>(a.y),
                      (const float*)a.rstd, a.M, a.N, m.chunks);
  });
}

// Row groups and the home of the per-row k values: the dgamma buffer when
// it holds M floats (it is written only by the final column reduction),
// else the workspace rows after the partials.
bool size_bwd_chunked(const BwdArgs& a, const DeviceInfo& d, Mapping* m, float** kbuf) {
  const int64_t cap = std::min<int64_t>(a.M, max_partials(d.sms));  // workspace rows
  int64_t RG = std::max<int64_t>(1, max_partials(d.sms) / m->chunks);
  if (a.M <= a.N) {
    *kbuf = a.dgamma;
  } else {
    const int64_t krows = (a.M + a.N - 1) / a.N;
    if (cap - krows < 1) return false;  // many short rows: not this mapping's shape
    RG = std::min<int64_t>(RG, cap - krows);
    *kbuf = a.ws + (cap - krows) * (int64_t)a.N;
  }
  RG = std::max<int64_t>(1, std::min<int64_t>(RG, cap));
  if (RG * m->chunks > INT32_MAX) return false;
  m->partials = RG;
  m->blocks = RG * m->chunks;
  return true;
}

cudaError_t launch_bwd_chunked(const BwdArgs& a, const Mapping& m, float* kbuf,
                               const DeviceInfo& d, cudaStream_t s) {
  return rmsk::with_types(a.dtype, a.gemma, a.dh != nullptr,
                         [&](auto* tp, auto* wp, auto gm, auto rs) -> cudaError_t {
    using T = std::remove_pointer_t<decltype(tp)>;
    using W = std::remove_pointer_t<decltype(wp)>;
    constexpr bool GEMMA = decltype(gm)::value;
    constexpr bool RES = decltype(rs)::value;
    const T* x = static_cast<const T*>(a.x);
    const T* dy = static_cast<const T*>(a.dy);
    const W* g = static_cast<const W*>(a.gamma);
    const int64_t rows_grid = std::min<int64_t>(a.M, (int64_t)d.sms * 4);
    cudaError_t e = rmsk::launch_pdl(rmsk::rms_rowstat_kernel<T, W, GEMMA, true, false>,
                               dim3((unsigned)rows_grid), dim3(rmsk::kChunkThreads), 0, s, x, dy,
                               g, a.rstd, kbuf, a.M, a.N, 0.f, (const T*)nullptr, (T*)nullptr);
    if (e != cudaSuccess) return e;
    return rmsk::launch_pdl(rmsk::rms_bwd_chunk_kernel<T, W, GEMMA, RES>, dim3((unsigned)m.blocks),
                      dim3(rmsk::kChunkThreads), 0, s, dy, x, g, a.rstd, (const float*)kbuf,
                      static_cast<T*>(a.dx), a.ws, a.M, a.N, m.chunks, m.partials,
                      static_cast<const T*>(a.dh));
  });
}

}  // namespace rmsi
