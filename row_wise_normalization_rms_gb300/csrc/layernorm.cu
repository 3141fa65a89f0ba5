// LayerNorm forward and backward on the same engine as RMSNorm.
//
//   mean = sum(x)/N,  var = sum((x - mean)^2)/N,  rstd = 1/sqrt(var + eps)
//   xhat = (x - mean)*rstd,  y = xhat*w + b            (one rounding per y)
//   g = dy*w,  c1 = sum(xhat*g)/N,  c2 = sum(g)/N,  dx = (g - (xhat*c1 + c2))*rstd
//   dw = sum over rows of dy*xhat,  db = sum over rows of dy
//
// Source: "第 07 章:LayerNorm——反向传播与原子锁", step 3 (forward: mean, then
// the variance of the centred values, mean and rstd saved) and § 3.0
// (backward: c1, c2, dx; dw and db as row contributions summed over rows).
// The chapter sums the contributions under grouped spin locks; here each
// persistent CTA keeps its column partials in registers across a static set
// of rows and writes one row of partials, and a fixed-order column
// reduction finishes dw and db: no atomics, no locks, deterministic.
//
// Mappings: the forward holds a row in registers (a thread group per row);
// the backward streams x and dy through a shared-memory ring filled by
// cp.async.bulk (bounded mbarrier waits, as the RMSNorm staged mapping);
// scalar kernels take any alignment.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace rmsk {

// Nonzero once a bounded wait in a LayerNorm kernel gave up.
__device__ int g_ln_device_status = 0;

// Sum over a group of G threads (G a multiple of 32; warps [first_warp,
// first_warp + G/32) of the CTA), every thread of the CTA calling: warp
// butterflies, one barrier, then each warp reduces the per-warp sums with a
// second butterfly, so all threads of the group get identical bits.  `red`
// holds one float per warp of the CTA.
__device__ __forceinline__ float ln_group_sum(float v, int G, int first_warp, float* red) {
  v = warp_sum(v);
  if (G == 32) return v;
  const int lane = threadIdx.x & 31;
  if (lane == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  return warp_sum(lane < (G >> 5) ? red[first_warp + lane] : 0.f);
}

// ---------------------------------------------------------------- forward

template <typename T, typename W, int KV>
__global__ void __launch_bounds__(1024)
ln_fwd_registers_kernel(const T* __restrict__ x, const W* __restrict__ w, const W* __restrict__ b,
                        T* __restrict__ y, float* __restrict__ mean_out,
                        float* __restrict__ rstd_out, int64_t M, int N, float inv_n, float eps,
                        int G) {
  using P = Pairs<T>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  constexpr int NP = P::n;
  __shared__ float red_a[32], red_b[32];
  const int NV = N / VN;
  const int grp = threadIdx.x / G;
  const int lig = threadIdx.x - grp * G;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / G) + grp;
  const bool active = row < M;
  const uint4* xr = reinterpret_cast<const uint4*>(x) + (active ? row : 0) * (int64_t)NV;
  pdl_trigger();
  pdl_wait();

  // The row is widened to float pairs once; the same registers then hold
  // the centred values x - mean.
  f32x2 xf[KV][NP];
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = lig + k * G;
    const uint4 q = (active && v < NV) ? ld_stream(xr + v) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < NP; ++i) xf[k][i] = P::get(q, i);
  }
  // mean
  f32x2 s2 = 0ull;
#pragma unroll
  for (int k = 0; k < KV; ++k)
#pragma unroll
    for (int i = 0; i < NP; ++i) s2 = add2(s2, xf[k][i]);
  const float mean = ln_group_sum(lo2(s2) + hi2(s2), G, grp * (G >> 5), red_a) * inv_n;
  // variance of the centred values (padding lanes and columns excluded)
  const f32x2 nm = splat2(-mean);
  f32x2 q2 = 0ull;
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = lig + k * G;
    if (active && v < NV) {
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        xf[k][i] = add2(xf[k][i], nm);
        q2 = fma2(xf[k][i], xf[k][i], q2);
      }
    }
  }
  const float var = ln_group_sum(lo2(q2) + hi2(q2), G, grp * (G >> 5), red_b) * inv_n;
  const float rstd = 1.0f / sqrtf(var + eps);
  if (!active) return;  // no barrier follows
  if (lig == 0) {
    mean_out[row] = mean;
    rstd_out[row] = rstd;
  }
  const f32x2 rr = splat2(rstd);
  uint4* yr = reinterpret_cast<uint4*>(y) + row * (int64_t)NV;
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = lig + k * G;
    if (v < NV) {
      const GV wv = GV::load(w, v);
      const GV bv = b != nullptr ? GV::load(b, v) : GV::zero();
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const f32x2 xh = mul2(xf[k][i], rr);
        const f32x2 yy = fma2(xh, wv.pair(i), bv.pair(i));  // + 0 without a bias
        if constexpr (sizeof(T) == 2) {
          o[i] = Half2Ops<T>::narrow(yy);
        } else {
          o[2 * i] = __float_as_uint(lo2(yy));
          o[2 * i + 1] = __float_as_uint(hi2(yy));
        }
      }
      st_stream(yr + v, make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
}

template <typename T, typename W>
__global__ void __launch_bounds__(256)
ln_fwd_scalar_kernel(const T* __restrict__ x, const W* __restrict__ w, const W* __restrict__ b,
                     T* __restrict__ y, float* __restrict__ mean_out, float* __restrict__ rstd_out,
                     int64_t M, int N, float inv_n, float eps) {
  using E = Elem<T>;
  __shared__ float red_a[8], red_b[8];
  const int64_t row = blockIdx.x;
  const T* xr = x + row * N;
  pdl_trigger();
  pdl_wait();
  // Compensated sums: a thread adds N / 256 terms in sequence.
  Kahan1 s;
  for (int j = threadIdx.x; j < N; j += 256) s.add(E::to_f(xr[j]));
  const float mean = group_sum(s.total(), 256, 0, red_a) * inv_n;
  Kahan1 q;
  for (int j = threadIdx.x; j < N; j += 256) {
    const float d = E::to_f(xr[j]) - mean;
    q.add(__fmul_rn(d, d));
  }
  const float rstd = 1.0f / sqrtf(group_sum(q.total(), 256, 0, red_b) * inv_n + eps);
  if (threadIdx.x == 0) {
    mean_out[row] = mean;
    rstd_out[row] = rstd;
  }
  T* yr = y + row * N;
  for (int j = threadIdx.x; j < N; j += 256) {
    const float xh = (E::to_f(xr[j]) - mean) * rstd;
    const float wj = Elem<W>::to_f(w[j]);
    yr[j] = E::from_f(b != nullptr ? fmaf(xh, wj, Elem<W>::to_f(b[j])) : xh * wj);
  }
}

// ---------------------------------------------------------------- backward

struct LnStagedParams {
  const void* x;
  const void* dy;
  const void* w;
  const float* mean;
  const float* rstd;
  void* dx;    // may equal dy
  float* wsw;  // [grid][N] dw partials
  float* wsb;  // [grid][N] db partials
  int64_t M;
  int N;
  float inv_n;  // 1/N rounded to float
  int G, R, S;
  int64_t ntiles;
  uint32_t tile_bytes, stage_bytes;
  long long wait_limit;
};

constexpr int kLnHeaderBytes = 1024;

// The backward over a ring of S stages of R rows (x then dy), like the
// RMSNorm staged mapping: first pass (row sums and column partials), one
// barrier, second pass (dx); a stage is refilled one barrier after its
// second pass.  Two row sums travel together (c1 and c2).
template <typename T, typename W, int KV>
__global__ void __launch_bounds__(512, 1)
ln_bwd_staged_kernel(const LnStagedParams p) {
  using P = Pairs<T>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  constexpr int NP = P::n;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  float2* red = reinterpret_cast<float2*>(smem + 64);                 // [2][32]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 576);  // [2]
  uint8_t* stages = smem + kLnHeaderBytes;

  const int NV = p.N / VN;
  const int q = threadIdx.x / p.G;
  const int lig = threadIdx.x - q * p.G;
  const int warp = threadIdx.x >> 5;
  const int first_warp = q * (p.G >> 5);
  const int nw = p.G >> 5;
  const int64_t my_tiles = (p.ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x;
  const int64_t row_bytes = (int64_t)p.N * sizeof(T);
  const uint32_t row_off = (uint32_t)(q * row_bytes);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.S; ++s) mbar_init(smem_u32(&full[s]), 1);
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();

  uint64_t pol = 0;
  int64_t issued = 0;  // thread 0 only
  int issue_stage = 0;  // issued % S, thread 0 only
  auto issue = [&](int64_t i) {
    const int64_t row0 = (blockIdx.x + i * gridDim.x) * p.R;
    const int64_t rows = min((int64_t)p.R, p.M - row0);
    const uint32_t bytes = (uint32_t)(rows * row_bytes);
    const int s = issue_stage;
    issue_stage = issue_stage + 1 == p.S ? 0 : issue_stage + 1;
    const uint32_t bar = smem_u32(&full[s]);
    const uint32_t dst = smem_u32(stages + (size_t)s * p.stage_bytes);
    mbar_arrive_expect_tx(bar, 2 * bytes);
    tma_load_1d(dst, static_cast<const char*>(p.x) + row0 * row_bytes, bytes, bar, pol);
    tma_load_1d(dst + p.tile_bytes, static_cast<const char*>(p.dy) + row0 * row_bytes, bytes, bar,
                pol);
  };
  if (threadIdx.x == 0) {
    pol = l2_evict_first_policy();
    const int64_t pre = min((int64_t)p.S, my_tiles);
    for (; issued < pre; ++issued) issue(issued);
  }

  // With four vectors per thread the weight is re-read through L1 at each
  // use (the partials already take 64 registers); otherwise it is held,
  // widened to float32 pairs once.
  constexpr bool kHoldW = KV < 4;
  // Re-read 16-bit weights meet dy as stored: g = dy*w by mixed-precision fma
  // (the same exact product), without widening either.
  constexpr bool kMixedG = !kHoldW && sizeof(T) == 2 && sizeof(W) == 2;
  f32x2 wf[kHoldW ? KV : 1][NP];
  f32x2 accw[KV][NP], accb[KV][NP];
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = lig + k * p.G;
    if (kHoldW) {
      const GV wk = v < NV ? GV::load(p.w, v) : GV::zero();
#pragma unroll
      for (int i = 0; i < NP; ++i) wf[k][i] = wk.pair(i);
    }
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      accw[k][i] = 0ull;
      accb[k][i] = 0ull;
    }
  }

  // The row statistics are fetched one tile ahead, off the critical path.
  // Rows advance by a fixed step; the stage and its parity are counters.
  const int64_t row_step = (int64_t)gridDim.x * p.R;
  int64_t row = (int64_t)blockIdx.x * p.R + q;
  auto stats = [&](int64_t t, int64_t rw, float& m, float& r) {
    m = 0.f;
    r = 0.f;
    if (t < my_tiles && rw < p.M) {
      m = p.mean[rw];
      r = p.rstd[rw];
    }
  };
  float mu_next, rs_next;
  stats(0, row, mu_next, rs_next);
  int s = 0;
  uint32_t parity = 0;
  int64_t i = 0;
  bool aborted = false;
  for (; i < my_tiles; ++i, row += row_step, s = (s + 1 == p.S) ? 0 : s + 1, parity ^= (s == 0)) {
    const int buf = (int)(i & 1);
    const bool active = row < p.M;
    const float mu = mu_next, rs = rs_next;
    stats(i + 1, row + row_step, mu_next, rs_next);
    if (!mbar_wait(smem_u32(&full[s]), parity, p.wait_limit)) abort_flag[buf] = 1;

    const uint32_t xs = smem_u32(stages + (size_t)s * p.stage_bytes) + row_off;
    const uint32_t ds = xs + p.tile_bytes;
    // xhat = x*rstd + (-mean*rstd): one fused multiply-add per element; its
    // rounding is within float32 steps of (|x| + |mean|)*rstd, as (x - mean)*rstd
    const f32x2 nmr = splat2(-mu * rs), rr = splat2(rs);
    f32x2 s1 = 0ull, s2 = 0ull;  // sum(xhat*g), sum(g)
    if (active) {
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int v = lig + k * p.G;
        if (v < NV) {
          const uint4 xq = lds128(xs + 16u * v), dq = lds128(ds + 16u * v);
          const GV wk = kHoldW ? GV::zero() : GV::load(p.w, v);
#pragma unroll
          for (int e = 0; e < NP; ++e) {
            const f32x2 xh = fma2(P::get(xq, e), rr, nmr);
            const f32x2 d = P::get(dq, e);
            f32x2 g;
            if constexpr (kHoldW) {
              g = mul2(d, wf[k][e]);
            } else if constexpr (kMixedG) {
              g = mul_exact2(word_of(dq, e), wk.word(e), (const T*)nullptr);
            } else {
              g = mul2(d, wk.pair(e));
            }
            s1 = fma2(xh, g, s1);
            s2 = add2(s2, g);
            accw[k][e] = fma2(d, xh, accw[k][e]);
            accb[k][e] = add2(accb[k][e], d);
          }
        }
      }
    }
    const float a1 = warp_sum(lo2(s1) + hi2(s1));
    const float a2 = warp_sum(lo2(s2) + hi2(s2));
    if ((threadIdx.x & 31) == 0) red[buf * 32 + warp] = make_float2(a1, a2);
    __syncthreads();  // sums visible; tile i-1 fully consumed
    if (abort_flag[buf]) {
      aborted = true;
      break;
    }
    if (threadIdx.x == 0 && i >= 1 && issued < my_tiles) issue(issued++);
    float t1, t2;
    {
      const int lane = threadIdx.x & 31;
      const float2 v = lane < nw ? red[buf * 32 + first_warp + lane] : make_float2(0.f, 0.f);
      t1 = warp_sum(v.x);
      t2 = warp_sum(v.y);
    }
    // dx = (g - (xhat*c1 + c2))*rstd = g*rstd + (xhat*c1r + c2r) with
    // c1r = -c1*rstd, c2r = -c2*rstd, and with xhat = x*rstd - mean*rstd
    // folded in: g*rstd + (x*ka + kb), ka = rstd*c1r, kb = -mean*rstd*c1r
    // + c2r (row constants; two fused multiply-adds an element pair).
    // x*ka + kb cancels like x - mean: its rounding stays within float32
    // steps of (|x| + |mean|)*rstd*|c1r| + |c2r|.
    const float c1r = -t1 * p.inv_n * rs, c2r = -t2 * p.inv_n * rs;
    const f32x2 ka = splat2(rs * c1r), kb = splat2(fmaf(-mu * rs, c1r, c2r));
    if (active) {
      uint4* out = reinterpret_cast<uint4*>(p.dx) + row * (int64_t)NV;
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int v = lig + k * p.G;
        if (v < NV) {
          const uint4 xq = lds128(xs + 16u * v), dq = lds128(ds + 16u * v);
          const GV wk = kHoldW ? GV::zero() : GV::load(p.w, v);
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < NP; ++e) {
            f32x2 g;
            if constexpr (kHoldW) {
              g = mul2(P::get(dq, e), wf[k][e]);
            } else if constexpr (kMixedG) {
              g = mul_exact2(word_of(dq, e), wk.word(e), (const T*)nullptr);
            } else {
              g = mul2(P::get(dq, e), wk.pair(e));
            }
            const f32x2 dxe = fma2(g, rr, fma2(P::get(xq, e), ka, kb));
            if constexpr (sizeof(T) == 2) {
              o[e] = Half2Ops<T>::narrow(dxe);
            } else {
              o[2 * e] = __float_as_uint(lo2(dxe));
              o[2 * e + 1] = __float_as_uint(hi2(dxe));
            }
          }
          st_stream(out + v, make_uint4(o[0], o[1], o[2], o[3]));
        }
      }
    }
  }
  if (aborted) {
    if (threadIdx.x == 0) {
      for (int64_t j = i; j < issued; ++j)
        mbar_wait(smem_u32(&full[j % p.S]), (uint32_t)((j / p.S) & 1), kDrainPolls);
      g_ln_device_status = 1;
      __threadfence();
    }
    return;
  }

  // One row of dw and one of db partials per CTA; groups of a CTA are
  // combined in group order through the idle stage memory.
  float* pw = p.wsw + (int64_t)blockIdx.x * p.N;
  float* pb = p.wsb + (int64_t)blockIdx.x * p.N;
  if (p.R == 1) {
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = lig + k * p.G;
      if (v < NV) {
        float4* w4 = reinterpret_cast<float4*>(pw + (int64_t)v * VN);
        float4* b4 = reinterpret_cast<float4*>(pb + (int64_t)v * VN);
#pragma unroll
        for (int c = 0; c < NP / 2; ++c) {
          w4[c] = make_float4(lo2(accw[k][2 * c]), hi2(accw[k][2 * c]), lo2(accw[k][2 * c + 1]),
                              hi2(accw[k][2 * c + 1]));
          b4[c] = make_float4(lo2(accb[k][2 * c]), hi2(accb[k][2 * c]), lo2(accb[k][2 * c + 1]),
                              hi2(accb[k][2 * c + 1]));
        }
      }
    }
  } else {
    float* part = reinterpret_cast<float*>(stages);  // [2][R][N] fits in the ring
    __syncthreads();
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = lig + k * p.G;
      if (v < NV) {
#pragma unroll
        for (int e = 0; e < NP; ++e) {
          const int64_t o = (int64_t)q * p.N + v * VN + 2 * e;
          part[o] = lo2(accw[k][e]);
          part[o + 1] = hi2(accw[k][e]);
          part[(int64_t)p.R * p.N + o] = lo2(accb[k][e]);
          part[(int64_t)p.R * p.N + o + 1] = hi2(accb[k][e]);
        }
      }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < p.N; j += blockDim.x) {
      float tw = 0.f, tb = 0.f;
      for (int qq = 0; qq < p.R; ++qq) {
        tw += part[(int64_t)qq * p.N + j];
        tb += part[(int64_t)(p.R + qq) * p.N + j];
      }
      pw[j] = tw;
      pb[j] = tb;
    }
  }
}

template <typename T, typename W>
__global__ void __launch_bounds__(256)
ln_bwd_scalar_kernel(const T* dy, const T* __restrict__ x, const W* __restrict__ w,
                     const float* __restrict__ mean, const float* __restrict__ rstd, T* dx,
                     float* __restrict__ wsw, float* __restrict__ wsb, int64_t M, int N,
                     float inv_n, int acc_in_smem) {
  using E = Elem<T>;
  __shared__ float red[2][2][8];
  // dw and db partials of this CTA, column j owned by thread j % 256: in
  // shared memory when 2N floats fit, else in the CTA's own workspace rows.
  extern __shared__ float acc_s[];
  float* accw = acc_in_smem ? acc_s : wsw + (int64_t)blockIdx.x * N;
  float* accb = acc_in_smem ? acc_s + N : wsb + (int64_t)blockIdx.x * N;
  pdl_wait();
  for (int j = threadIdx.x; j < N; j += 256) {
    accw[j] = 0.f;
    accb[j] = 0.f;
  }
  int it = 0;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x, ++it) {
    const T* xr = x + row * N;
    const T* dr = dy + row * N;
    const float mu = mean[row], rs = rstd[row];
    Kahan1 s1, s2;
    for (int j = threadIdx.x; j < N; j += 256) {
      const float xh = (E::to_f(xr[j]) - mu) * rs;
      const float d = E::to_f(dr[j]);
      const float g = d * Elem<W>::to_f(w[j]);
      s1.add(__fmul_rn(xh, g));
      s2.add(g);
      accw[j] = fmaf(d, xh, accw[j]);
      accb[j] += d;
    }
    const float c1 = group_sum(s1.total(), 256, 0, red[it & 1][0]) * inv_n;
    const float c2 = group_sum(s2.total(), 256, 0, red[it & 1][1]) * inv_n;
    T* out = dx + row * N;
    for (int j = threadIdx.x; j < N; j += 256) {
      const float xh = (E::to_f(xr[j]) - mu) * rs;
      const float g = E::to_f(dr[j]) * Elem<W>::to_f(w[j]);
      out[j] = E::from_f((g - fmaf(xh, c1, c2)) * rs);
    }
  }
  if (acc_in_smem) {
    for (int j = threadIdx.x; j < N; j += 256) {
      wsw[(int64_t)blockIdx.x * N + j] = accw[j];
      wsb[(int64_t)blockIdx.x * N + j] = accb[j];
    }
  }
}

}  // namespace rmsk

namespace rmsi {

namespace {

template <typename F>
cudaError_t with_types(int dtype, F&& f) {
  switch (dtype) {
    case kBF16: return f((__nv_bfloat16*)nullptr, (__nv_bfloat16*)nullptr);
    case kF16: return f((__half*)nullptr, (__half*)nullptr);
    case kBF16W32: return f((__nv_bfloat16*)nullptr, (float*)nullptr);
    case kF16W32: return f((__half*)nullptr, (float*)nullptr);
    default: return f((float*)nullptr, (float*)nullptr);
  }
}

struct LnOcc {
  const void* k;
  int dev, threads;
  size_t smem;
  int occ;
};
std::mutex g_ln_mu;
LnOcc g_ln_occ[64];
int g_ln_n = 0;

cudaError_t ln_occupancy(const void* k, const DeviceInfo& d, int threads, size_t smem, int* occ) {
  std::lock_guard<std::mutex> lk(g_ln_mu);
  for (int i = 0; i < g_ln_n; ++i)
    if (g_ln_occ[i].k == k && g_ln_occ[i].dev == d.device && g_ln_occ[i].threads == threads &&
        g_ln_occ[i].smem == smem) {
      *occ = g_ln_occ[i].occ;
      return cudaSuccess;
    }
  cudaError_t e = opt_in_max_smem(k, d);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, threads, smem);
  if (e != cudaSuccess) return e;
  if (g_ln_n < 64) g_ln_occ[g_ln_n++] = LnOcc{k, d.device, threads, smem, *occ};
  return cudaSuccess;
}

}  // namespace

// Backward rows of up to this many 16-byte vectors take two vectors per
// thread (twice the threads a row, weights held in registers) instead of
// four: GB300, M = 4096 fp16, N = 1024 17.4 -> 14.4 us and N = 4096 34.1 ->
// 33.4 us per call; from N = 8192 four are faster (52.4 against 54.6 us).
#ifndef RMS_LN_BWD_KV2_MAX_NV
#define RMS_LN_BWD_KV2_MAX_NV 512
#endif
// Most threads a backward CTA takes for its rows.
#ifndef RMS_LN_BWD_MAX_CTA_THREADS
#define RMS_LN_BWD_MAX_CTA_THREADS 256
#endif
#ifndef RMS_LN_FWD_CTA_THREADS
#define RMS_LN_FWD_CTA_THREADS 128
#endif
bool ln_plan(int N, int dtype, bool bwd, int path, bool aligned, const DeviceInfo& d, Mapping* m,
             int64_t M) {
  const int b = dtype_bytes(dtype);
  const int64_t row_bytes = (int64_t)N * b;
  const int NV = (int)(row_bytes / 16);
  const bool vec_ok = aligned && row_bytes % 16 == 0;
  if (!bwd && (path == kAuto || path == kRegisters) && vec_ok) {
    int kv = NV <= 32 ? 1 : NV <= 64 ? 2 : 4;
    int G = kv < 4 ? 32 : ((NV + 3) / 4 + 31) / 32 * 32;
    if (G <= 1024) {
      m->path = kRegisters;
      m->kv = kv;
      m->G = G;
      // One 128-thread row a CTA rather than two in 256 threads (GB300: 4096
      // x 4096 f16 15.9 -> 14.5 us, 32768 x 4096 91.3 -> 86.2 us); rows of
      // a warp or less still share 256-thread CTAs.
      const int cta = G >= 64 ? RMS_LN_FWD_CTA_THREADS : 256;
      m->rows_per_cta = G >= cta ? 1 : cta / G;
      m->threads = G * m->rows_per_cta;
      m->smem = 0;
      return true;
    }
  }
  if (bwd && (path == kAuto || path == kStaged) && vec_ok) {
    // At most four vectors per thread: the dw and db partials of a thread's
    // columns live in registers (at most 128 a thread).  CTAs of up to 256
    // threads (two per SM) where the row allows, else one row of up to 512
    // threads (32 KiB rows) and one CTA per SM.
    const int kv = NV <= 32 ? 1 : NV <= RMS_LN_BWD_KV2_MAX_NV ? 2 : 4;
    const int G = ((NV + kv - 1) / kv + 31) / 32 * 32;
    if (G <= 512) {
      int R = (int)(16384 / row_bytes);
      R = std::max(1, std::min(R, 16));
      while (R > 1 && G * R > RMS_LN_BWD_MAX_CTA_THREADS) --R;
      // Halve the tile while the persistent CTAs (two per SM at 256 threads,
      // four at 128, by registers) would get fewer than 20 tiles each (a
      // ragged last wave), down to 8 KiB a tensor (smaller tiles cost more
      // per row than the tail they save).
      const int per_sm = (RMS_LN_BWD_MAX_CTA_THREADS <= 128 && G * R <= 128) ? 4
                         : G * R <= 256 ? 2 : 1;
      const int64_t ctas = (int64_t)per_sm * d.sms;
      while (R > 1 && (R / 2) * row_bytes >= 8192 && M > 0 && (M + R - 1) / R < 20 * ctas)
        R /= 2;
      const int64_t stage = 2 * (int64_t)R * row_bytes;
      const int64_t budget = 224 * 1024, cap = (int64_t)d.smem_optin - rmsk::kLnHeaderBytes;
      int cps = 0, S = 0;
      for (int c = 4; c >= 1; --c) {
        const int64_t per = std::min(budget / c, cap);
        if (3 * stage <= per) {
          cps = c;
          S = (int)std::min<int64_t>(8, per / stage);
          break;
        }
      }
      if (cps > 0) {
        m->path = kStaged;
        m->kv = kv;
        m->G = G;
        m->rows_per_cta = R;
        m->threads = G * R;
        m->stages = S;
        m->smem = rmsk::kLnHeaderBytes + (size_t)S * stage;
        m->blocks = cps;
        return true;
      }
    }
  }
  if (path == kAuto || path == kScalar) {
    m->path = kScalar;
    m->G = m->threads = 256;
    m->rows_per_cta = 1;
    m->smem = bwd ? (size_t)2 * N * sizeof(float) : 0;
    m->smem_acc = 1;
    if (m->smem + 1024 > d.smem_optin) {
      m->smem = 0;  // too wide: accumulate in the workspace rows instead
      m->smem_acc = 0;
    }
    return true;
  }
  return false;
}

cudaError_t ln_launch_fwd(const LnFwdArgs& a, const Mapping& m, cudaStream_t s) {
  return with_types(a.dtype, [&](auto* tp, auto* wp) -> cudaError_t {
    using T = std::remove_pointer_t<decltype(tp)>;
    using W = std::remove_pointer_t<decltype(wp)>;
    const T* x = static_cast<const T*>(a.x);
    const W* w = static_cast<const W*>(a.w);
    const W* b = static_cast<const W*>(a.b);
    T* y = static_cast<T*>(a.y);
    const float inv_n = (float)(1.0 / a.N);
    if (m.path == kRegisters) {
      const dim3 grid((unsigned)((a.M + m.rows_per_cta - 1) / m.rows_per_cta)), block(m.threads);
      switch (m.kv) {
        case 1: return rmsk::launch_pdl(rmsk::ln_fwd_registers_kernel<T, W, 1>, grid, block, 0, s, x, w, b, y, a.mean, a.rstd, a.M, a.N, inv_n, a.eps, m.G);
        case 2: return rmsk::launch_pdl(rmsk::ln_fwd_registers_kernel<T, W, 2>, grid, block, 0, s, x, w, b, y, a.mean, a.rstd, a.M, a.N, inv_n, a.eps, m.G);
        default: return rmsk::launch_pdl(rmsk::ln_fwd_registers_kernel<T, W, 4>, grid, block, 0, s, x, w, b, y, a.mean, a.rstd, a.M, a.N, inv_n, a.eps, m.G);
      }
    }
    return rmsk::launch_pdl(rmsk::ln_fwd_scalar_kernel<T, W>, dim3((unsigned)a.M), dim3(256), 0, s,
                            x, w, b, y, a.mean, a.rstd, a.M, a.N, inv_n, a.eps);
  });
}

cudaError_t ln_size_bwd(const LnBwdArgs& a, const DeviceInfo& d, Mapping* m) {
  return with_types(a.dtype, [&](auto* tp, auto* wp) -> cudaError_t {
    using T = std::remove_pointer_t<decltype(tp)>;
    using W = std::remove_pointer_t<decltype(wp)>;
    const void* k;
    if (m->path == kStaged) {
      k = m->kv == 1   ? reinterpret_cast<const void*>(&rmsk::ln_bwd_staged_kernel<T, W, 1>)
          : m->kv == 2 ? reinterpret_cast<const void*>(&rmsk::ln_bwd_staged_kernel<T, W, 2>)
                       : reinterpret_cast<const void*>(&rmsk::ln_bwd_staged_kernel<T, W, 4>);
    } else {
      k = reinterpret_cast<const void*>(&rmsk::ln_bwd_scalar_kernel<T, W>);
    }
    int occ = 0;
    cudaError_t e;
    if (m->path == kStaged) {
      // CTAs per SM as registers allow (with the smallest ring), then the
      // deepest ring that many CTAs can share.
      const int64_t stage = (int64_t)m->smem - rmsk::kLnHeaderBytes;
      const int64_t one = stage / m->stages;
      e = ln_occupancy(k, d, m->threads, rmsk::kLnHeaderBytes + 3 * one, &occ);
      if (e != cudaSuccess) return e;
      if (occ < 1) return cudaErrorInvalidConfiguration;
      const int cps = std::min<int>(occ, m->blocks);
      const int64_t per = std::min<int64_t>(224 * 1024 / cps,
                                            (int64_t)d.smem_optin - rmsk::kLnHeaderBytes);
      m->stages = (int)std::max<int64_t>(3, std::min<int64_t>(8, per / one));
      m->smem = rmsk::kLnHeaderBytes + (size_t)m->stages * one;
      m->blocks = cps;
    }
    e = ln_occupancy(k, d, m->threads, m->smem, &occ);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int64_t per_sm = m->path == kStaged ? std::min<int64_t>(occ, m->blocks) : occ;
    int64_t P = per_sm * d.sms;
    if (P > max_partials(d.sms)) P = max_partials(d.sms);
    const int64_t units = (a.M + m->rows_per_cta - 1) / m->rows_per_cta;
    if (P > units) P = units;
    if (P < 1) P = 1;
    m->blocks = P;
    m->partials = P;
    return cudaSuccess;
  });
}

cudaError_t ln_launch_bwd(const LnBwdArgs& a, const Mapping& m, long long wait_limit,
                          cudaStream_t s) {
  return with_types(a.dtype, [&](auto* tp, auto* wp) -> cudaError_t {
    using T = std::remove_pointer_t<decltype(tp)>;
    using W = std::remove_pointer_t<decltype(wp)>;
    if (m.path == kStaged) {
      rmsk::LnStagedParams p{};
      p.x = a.x;
      p.dy = a.dy;
      p.w = a.w;
      p.mean = a.mean;
      p.rstd = a.rstd;
      p.dx = a.dx;
      p.wsw = a.wsw;
      p.wsb = a.wsb;
      p.M = a.M;
      p.N = a.N;
      p.inv_n = (float)(1.0 / a.N);
      p.G = m.G;
      p.R = m.rows_per_cta;
      p.S = m.stages;
      p.ntiles = (a.M + p.R - 1) / p.R;
      p.tile_bytes = (uint32_t)((int64_t)p.R * a.N * sizeof(T));
      p.stage_bytes = 2 * p.tile_bytes;
      p.wait_limit = wait_limit;
      const dim3 grid((unsigned)m.blocks), block(m.threads);
      if (m.kv == 1)
        return rmsk::launch_pdl(rmsk::ln_bwd_staged_kernel<T, W, 1>, grid, block, m.smem, s, p);
      if (m.kv == 2)
        return rmsk::launch_pdl(rmsk::ln_bwd_staged_kernel<T, W, 2>, grid, block, m.smem, s, p);
      return rmsk::launch_pdl(rmsk::ln_bwd_staged_kernel<T, W, 4>, grid, block, m.smem, s, p);
    }
    return rmsk::launch_pdl(rmsk::ln_bwd_scalar_kernel<T, W>, dim3((unsigned)m.blocks), dim3(256),
                            m.smem, s, static_cast<const T*>(a.dy), static_cast<const T*>(a.x),
                            static_cast<const W*>(a.w), a.mean, a.rstd, static_cast<T*>(a.dx),
                            a.wsw, a.wsb, a.M, a.N, (float)(1.0 / a.N), m.smem_acc);
  });
}

cudaError_t take_ln_device_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, rmsk::g_ln_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(rmsk::g_ln_device_status, &zero, sizeof(int));
    if (e != cudaSuccess) return e;
  }
  *status = v;
  return cudaSuccess;
}

}  // namespace rmsi
