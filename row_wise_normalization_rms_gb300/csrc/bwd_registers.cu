// Backward RMSNorm, register mapping, persistent grid.
//
// A group of G threads owns one row at a time and holds x, dy and the
// weight in registers as 16-byte vectors:
//
//   u  = dy * g                    (g = gamma, or 1 + gamma for Gemma)
//   c  = sum(u * x) / N            (the true N)
//   dx = r * u - x * r^3 * c       (r is the forward's saved rstd)
//
// dx is stored to dx, or over dy when the caller asks for it in place (the
// whole row is already in registers when it is overwritten).  The weight
// gradient is a sum over rows, so each thread also accumulates
// dy * x * r for the columns it owns, across every row its group visits.
// Rows are dealt to groups statically (row = group id + k * groups), and at
// the end each CTA writes one float32 row of column partials to the
// workspace (groups of a CTA are combined in group order through shared
// memory).  A second kernel sums the partial rows in a fixed order.  No
// atomics and no locks: the result depends only on M, N and the grid size.
//
// Sources: "Hướng dẫn Triton RMSNorm: kernel, backward…", sections "Vì sao
// cần một lượt đi và một lượt về?", "Backward đầu vào: giữ đúng N",
// "Reduce dgamma không có race khi ghi", "Tổng không phải trung bình";
// "02 · 手写 Triton kernel:RMSNorm / RoPE / SwiGLU", section 3 (dx into dy).
#include "common.cuh"
#include "internal.h"

namespace rmsk {

// With RES, dh (the gradient reaching the same input through a residual
// path; it may be the dx buffer itself) is added to dx before its rounding.
template <typename T, typename W, int KV, bool GEMMA, bool RES>
__global__ void __launch_bounds__(512)
rms_bwd_registers_kernel(const T* dy, const T* __restrict__ x, const W* __restrict__ gamma,
                         const float* __restrict__ rstd, T* dx, float* __restrict__ ws, int64_t M,
                         int N, int G, const T* dh) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  constexpr int NP = Math::kPairs;
  __shared__ float red[2][16];
  extern __shared__ float part[];  // [R][N] when R > 1 groups share the CTA

  const int NV = N / VN;
  const int R = blockDim.x / G;
  const int grp = threadIdx.x / G;
  const int lig = threadIdx.x - grp * G;
  const int64_t groups = (int64_t)gridDim.x * R;
  const int64_t gid0 = (int64_t)blockIdx.x * R;  // the CTA's first group: it has the most rows
  const int64_t gid = gid0 + grp;
  const int64_t iters = gid0 < M ? (M - gid0 + groups - 1) / groups : 0;
  // Let the column reduction (a programmatic dependent) launch into SMs this
  // grid frees; it waits for this grid's completion before reading.
  pdl_wait();

  GV gw[KV];
  f32x2 acc[KV][NP];
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = lig + k * G;
    gw[k] = v < NV ? GV::load(gamma, v) : GV::zero();
#pragma unroll
    for (int i = 0; i < NP; ++i) acc[k][i] = 0ull;
  }

  // x, dy and r of the group's row of iteration `i` (zeros past the rows).
  auto fetch = [&](int64_t i, uint4 (&xa)[KV], uint4 (&da)[KV], float& ra) {
    const int64_t rw = gid + i * groups;
    const bool act = i < iters && rw < M;
    const int64_t b = (act ? rw : 0) * (int64_t)NV;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = lig + k * G;
      const bool in = act && v < NV;
      xa[k] = in ? ld_stream(reinterpret_cast<const uint4*>(x) + b + v) : make_uint4(0u, 0u, 0u, 0u);
      da[k] = in ? ld_stream(reinterpret_cast<const uint4*>(dy) + b + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    ra = act ? rstd[rw] : 0.f;
  };
  // Narrow rows fetch the next row while the current one is reduced and
  // written: its loads overlap the group's arithmetic instead of following
  // it (GB300, 1 KiB bf16 rows: 81 -> 91 % of HBM).  Not for float32 rows of
  // two vectors a thread, where the extra registers cost occupancy (98 -> 91 %).
  constexpr bool kPrefetch = KV == 1 || (KV == 2 && sizeof(T) == 2);
  uint4 xn[kPrefetch ? KV : 1], dn[kPrefetch ? KV : 1];
  float rn = 0.f;
  if constexpr (kPrefetch) fetch(0, xn, dn, rn);

  for (int64_t it = 0; it < iters; ++it) {
    const int64_t row = gid + it * groups;
    const bool active = row < M;
    const int64_t base = (active ? row : 0) * (int64_t)NV;
    uint4 xv[KV], dv[KV];
    float r;
    if constexpr (kPrefetch) {
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        xv[k] = xn[k];
        dv[k] = dn[k];
      }
      r = rn;
      fetch(it + 1, xn, dn, rn);
    } else {
      fetch(it, xv, dv, r);
    }

    // Zero vectors (inactive rows, columns past N) add nothing to either sum.
    f32x2 sux2 = 0ull;
#pragma unroll
    for (int k = 0; k < KV; ++k) Math::backward_sums(xv[k], dv[k], gw[k], r, sux2, acc[k]);
    uint4 hv[RES ? KV : 1];  // fetched while the row sum is reduced
    if (RES) {
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int v = lig + k * G;
        hv[k] = (active && v < NV) ? ld_stream(reinterpret_cast<const uint4*>(dh) + base + v)
                                   : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    const float sux = (KV == 1 && G < 32)
                          ? lane_group_sum(lo2(sux2) + hi2(sux2), G)
                          : group_sum(lo2(sux2) + hi2(sux2), G, grp * (G >> 5), red[it & 1]);
    const float kc = sux / (float)N;  // r * mean(u*x)

    if (active) {
      uint4* out = reinterpret_cast<uint4*>(dx) + base;
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int v = lig + k * G;
        if (v < NV)
          st_stream(out + v, RES ? Math::backward_dx_add(xv[k], dv[k], gw[k], r, kc, hv[RES ? k : 0])
                                 : Math::backward_dx(xv[k], dv[k], gw[k], r, kc));
      }
    }
  }

  // One workspace row per CTA: this CTA's column partial sums.
  float* wp = ws + (int64_t)blockIdx.x * N;
  if (R == 1) {
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = lig + k * G;
      if (v < NV) {
        float4* w4 = reinterpret_cast<float4*>(wp + (int64_t)v * VN);
#pragma unroll
        for (int q = 0; q < NP / 2; ++q)
          w4[q] = make_float4(lo2(acc[k][2 * q]), hi2(acc[k][2 * q]), lo2(acc[k][2 * q + 1]),
                              hi2(acc[k][2 * q + 1]));
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = lig + k * G;
      if (v < NV) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          part[(int64_t)grp * N + v * VN + 2 * i] = lo2(acc[k][i]);
          part[(int64_t)grp * N + v * VN + 2 * i + 1] = hi2(acc[k][i]);
        }
      }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < N; j += blockDim.x) {
      float t = 0.f;
      for (int q = 0; q < R; ++q) t += part[(int64_t)q * N + j];
      wp[j] = t;
    }
  }
}

template <typename T, typename W, int KV, bool RES>
static const void* kernel_ptr(bool gemma) {
  return gemma ? reinterpret_cast<const void*>(&rms_bwd_registers_kernel<T, W, KV, true, RES>)
               : reinterpret_cast<const void*>(&rms_bwd_registers_kernel<T, W, KV, false, RES>);
}

template <typename T, typename W>
static const void* pick(int kv, bool gemma, bool res) {
  switch (kv) {
    case 1: return res ? kernel_ptr<T, W, 1, true>(gemma) : kernel_ptr<T, W, 1, false>(gemma);
    case 2: return res ? kernel_ptr<T, W, 2, true>(gemma) : kernel_ptr<T, W, 2, false>(gemma);
    case 4: return res ? kernel_ptr<T, W, 4, true>(gemma) : kernel_ptr<T, W, 4, false>(gemma);
    default: return nullptr;
  }
}

template <typename T, typename W, bool GEMMA, bool RES>
static cudaError_t launch_g(const rmsi::BwdArgs& a, const rmsi::Mapping& m, cudaStream_t s) {
  const dim3 grid((unsigned)m.blocks), block(m.threads);
  const T* dy = static_cast<const T*>(a.dy);
  const T* x = static_cast<const T*>(a.x);
  const W* g = static_cast<const W*>(a.gamma);
  T* dx = static_cast<T*>(a.dx);
  const T* dh = static_cast<const T*>(a.dh);
  switch (m.kv) {
    case 1: return launch_pdl(rms_bwd_registers_kernel<T, W, 1, GEMMA, RES>, grid, block, m.smem, s, dy, x, g, a.rstd, dx, a.ws, a.M, a.N, m.G, dh);
    case 2: return launch_pdl(rms_bwd_registers_kernel<T, W, 2, GEMMA, RES>, grid, block, m.smem, s, dy, x, g, a.rstd, dx, a.ws, a.M, a.N, m.G, dh);
    case 4: return launch_pdl(rms_bwd_registers_kernel<T, W, 4, GEMMA, RES>, grid, block, m.smem, s, dy, x, g, a.rstd, dx, a.ws, a.M, a.N, m.G, dh);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, typename W>
static cudaError_t launch_t(const rmsi::BwdArgs& a, const rmsi::Mapping& m, cudaStream_t s) {
  if (a.dh) return a.gemma ? launch_g<T, W, true, true>(a, m, s) : launch_g<T, W, false, true>(a, m, s);
  return a.gemma ? launch_g<T, W, true, false>(a, m, s) : launch_g<T, W, false, false>(a, m, s);
}

}  // namespace rmsk

namespace rmsi {

cudaError_t size_bwd_registers(const BwdArgs& a, const DeviceInfo& d, Mapping* m) {
  m->smem = m->rows_per_cta > 1 ? (size_t)m->rows_per_cta * a.N * sizeof(float) : 0;
  const void* k;
  switch (a.dtype) {
    case kBF16: k = rmsk::pick<__nv_bfloat16, __nv_bfloat16>(m->kv, a.gemma, a.dh != nullptr); break;
    case kF16: k = rmsk::pick<__half, __half>(m->kv, a.gemma, a.dh != nullptr); break;
    case kBF16W32: k = rmsk::pick<__nv_bfloat16, float>(m->kv, a.gemma, a.dh != nullptr); break;
    case kF16W32: k = rmsk::pick<__half, float>(m->kv, a.gemma, a.dh != nullptr); break;
    default: k = rmsk::pick<float, float>(m->kv, a.gemma, a.dh != nullptr); break;
  }
  if (!k) return cudaErrorInvalidValue;
  int occ = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, m->threads, m->smem);
  if (e != cudaSuccess) return e;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  int64_t P = (int64_t)occ * d.sms;
  if (P > max_partials(d.sms)) P = max_partials(d.sms);
  const int64_t need = (a.M + m->rows_per_cta - 1) / m->rows_per_cta;
  if (P > need) P = need;
  if (P < 1) P = 1;
  m->blocks = P;
  m->partials = P;
  return cudaSuccess;
}

cudaError_t launch_bwd_registers(const BwdArgs& a, const Mapping& m, cudaStream_t s) {
  switch (a.dtype) {
    case kBF16: return rmsk::launch_t<__nv_bfloat16, __nv_bfloat16>(a, m, s);
    case kF16: return rmsk::launch_t<__half, __half>(a, m, s);
    case kBF16W32: return rmsk::launch_t<__nv_bfloat16, float>(a, m, s);
    case kF16W32: return rmsk::launch_t<__half, float>(a, m, s);
    default: return rmsk::launch_t<float, float>(a, m, s);
  }
}

}  // namespace rmsi
