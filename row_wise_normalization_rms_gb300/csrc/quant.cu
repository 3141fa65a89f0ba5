// RMSNorm forward with the output quantised to FP8 (E4M3) for the GEMM that
// consumes it, in the same kernel: y never reaches memory in the activation
// type, only its 1-byte codes and one float32 scale per row.
//
//   y    = the forward's y, with the forward's roundings (the stored value)
//   amax = max_j |y_j|,  s = amax / 448,  q_j = e4m3(y_j * (448 / amax))
//   (round to nearest even, saturating at +-448; a zero row gets s = 1)
//
// Source for y: "Hướng dẫn Triton RMSNorm: kernel, backward…", section "Vấn
// đề và công thức tham chiếu", and the cast order of "02 · 手写 Triton
// kernel:RMSNorm / RoPE / SwiGLU", section 3.  The fusion (an elementwise
// neighbour kept in registers, each tensor read or written once) is that
// page's sections 1-2; the E4M3 format and the per-row absolute-maximum
// scale are the plain reading of "quantise y for the next GEMM".
#include <type_traits>

#include "common.cuh"
#include "e4m3.cuh"
#include "internal.h"

namespace rmsk {

// Max over a warp in one instruction (the warp-wide float32 max reduction;
// like fmaxf it ignores NaN operands).
__device__ __forceinline__ float warp_max(float v) {
  float m;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(v));
  return m;
}

// Max over a group of G threads (as group_sum; max is order-free).
__device__ __forceinline__ float group_max(float v, int G, int first_warp, float* red) {
  if (G < 32) {
    for (int o = G >> 1; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
  }
  v = warp_max(v);
  if (G == 32) return v;
  const int lane = threadIdx.x & 31;
  if (lane == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  return warp_max(lane < (G >> 5) ? red[first_warp + lane] : 0.f);
}

// Row in registers (the register forward's mapping, at most 512 threads a
// CTA, two CTAs an SM at least): r, y, amax, codes.
template <typename T, typename W, int KV, bool GEMMA>
__global__ void __launch_bounds__(512, 2)
rms_fwd_quant_registers_kernel(const T* __restrict__ x, const W* __restrict__ gamma,
                               uint8_t* __restrict__ q, float* __restrict__ scale,
                               float* __restrict__ rstd, int64_t M, int N, float eps, int G) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  using P = Pairs<T>;
  constexpr int VN = Elem<T>::kPerVec;
  constexpr int NP = P::n;
  __shared__ float red_s[32], red_m[32];
  const int NV = N / VN;
  const int grp = threadIdx.x / G;
  const int lig = threadIdx.x - grp * G;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / G) + grp;
  const bool active = row < M;
  const uint4* xr = reinterpret_cast<const uint4*>(x) + (active ? row : 0) * (int64_t)NV;
  pdl_trigger();
  pdl_wait();

  uint4 v[KV];
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int j = lig + k * G;
    v[k] = (active && j < NV) ? ld_stream(xr + j) : make_uint4(0u, 0u, 0u, 0u);
  }
  float ss_lo = 0.f, ss_hi = 0.f;
#pragma unroll
  for (int k = 0; k < KV; ++k) SumSqDirect<T>::add(v[k], ss_lo, ss_hi);
  const float ss = G < 32 ? lane_group_sum(ss_lo + ss_hi, G)
                                       : group_sum(ss_lo + ss_hi, G, grp * (G >> 5), red_s);
  const float r = 1.0f / sqrtf(ss / (float)N + eps);
  // y as the forward stores it, in place of x; its absolute maximum
  AbsMax<T> am;
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int j = lig + k * G;
    if (active && j < NV) {
      v[k] = Math::forward(v[k], GV::load(gamma, j), r);
      am.add(v[k]);
    }
  }
  const float amax = group_max(am.value(), G, grp * (G >> 5), red_m);
  if (!active) return;  // no barrier follows
  const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 1.0f;
  if (lig == 0) {
    rstd[row] = r;
    scale[row] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  }
  uint8_t* qr = q + row * (int64_t)N;
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int j = lig + k * G;
    if (j < NV) {
      uint32_t c[NP];
      const f32x2 iv = splat2(inv);
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const f32x2 p = mul2(stored_pair<T>(v[k], i), iv);
        c[i] = f2_to_e4m3x2(lo2(p), hi2(p));
      }
      if constexpr (NP == 4) {  // 8 codes
        *reinterpret_cast<uint2*>(qr + (int64_t)j * VN) =
            make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
      } else {  // 4 codes
        *reinterpret_cast<uint32_t*>(qr + (int64_t)j * VN) = c[0] | (c[1] << 16);
      }
    }
  }
}

// The same row in registers with half the threads: each thread holds the
// vectors of two of the register forward's threads (Gv threads of four
// vectors a row; here G = Gv/2 rounded up to a warp, real thread t standing
// for t and t + G), so every per-row step (the reductions, the square root,
// the scale's division) is issued by half the warps.  The sum of squares
// keeps the register forward's order exactly: each stood-for thread's
// chain, then each stood-for warp's butterfly, then the Gv/32 warp sums in
// order.  r, and so y, equal rms_fwd's bit for bit.
template <typename T, typename W, bool GEMMA>
__global__ void __launch_bounds__(256, 4)
rms_fwd_quant_pairs_kernel(const T* __restrict__ x, const W* __restrict__ gamma,
                           uint8_t* __restrict__ q, float* __restrict__ scale,
                           float* __restrict__ rstd, int64_t M, int N, float eps, int G, int Gv) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  using P = Pairs<T>;
  constexpr int VN = Elem<T>::kPerVec;
  constexpr int NP = P::n;
  __shared__ float red_s[32], red_m[32];
  const int NV = N / VN;
  const int grp = threadIdx.x / G;
  const int lig = threadIdx.x - grp * G;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / G) + grp;
  const bool active = row < M;
  const uint4* xr = reinterpret_cast<const uint4*>(x) + (active ? row : 0) * (int64_t)NV;
  pdl_trigger();
  pdl_wait();

  // v[2k + h]: vector k of stood-for thread u_h = lig + h*G, column u_h + k*Gv
  uint4 v[8];
  bool ok[8];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int u = lig + h * G;
      const int j = u + k * Gv;
      ok[2 * k + h] = active && u < Gv && j < NV;
      v[2 * k + h] = ok[2 * k + h] ? ld_stream(xr + j) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  float s_lo[2] = {0.f, 0.f}, s_hi[2] = {0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int h = 0; h < 2; ++h) SumSqDirect<T>::add(v[2 * k + h], s_lo[h], s_hi[h]);
  }
  const int nw = G >> 5;              // real warps of a row
  const int base = grp * 2 * nw;      // this row's slots: stood-for warps 0 .. 2*nw-1
  const int w = (threadIdx.x >> 5) - grp * nw;
  const float a0 = warp_sum(s_lo[0] + s_hi[0]);
  const float a1 = warp_sum(s_lo[1] + s_hi[1]);
  if ((threadIdx.x & 31) == 0) {
    red_s[base + w] = a0;
    red_s[base + nw + w] = a1;
  }
  __syncthreads();
  float ss = 0.f;
  for (int i = 0; i < (Gv >> 5); ++i) ss += red_s[base + i];
  const float r = 1.0f / sqrtf(ss / (float)N + eps);
  // y as the forward stores it, in place of x; its absolute maximum
  AbsMax<T> am;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int j = lig + (i & 1) * G + (i >> 1) * Gv;
    if (ok[i]) {
      v[i] = Math::forward(v[i], GV::load(gamma, j), r);
      am.add(v[i]);
    }
  }
  const float amax = group_max(am.value(), G, grp * nw, red_m);
  if (!active) return;  // no barrier follows
  const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 1.0f;
  if (lig == 0) {
    rstd[row] = r;
    scale[row] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  }
  uint8_t* qr = q + row * (int64_t)N;
  const f32x2 iv = splat2(inv);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int j = lig + (i & 1) * G + (i >> 1) * Gv;
    if (ok[i]) {
      uint32_t c[NP];
#pragma unroll
      for (int e = 0; e < NP; ++e) {
        const f32x2 p = mul2(stored_pair<T>(v[i], e), iv);
        c[e] = f2_to_e4m3x2(lo2(p), hi2(p));
      }
      if constexpr (NP == 4) {  // 8 codes
        *reinterpret_cast<uint2*>(qr + (int64_t)j * VN) =
            make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
      } else {  // 4 codes
        *reinterpret_cast<uint32_t*>(qr + (int64_t)j * VN) = c[0] | (c[1] << 16);
      }
    }
  }
}

// Any alignment and width: one CTA per row, the row read three times (sum
// of squares, absolute maximum of y, codes); element for element the same
// roundings as the scalar forward.
template <typename T, typename W>
__global__ void __launch_bounds__(256)
rms_fwd_quant_scalar_kernel(const T* __restrict__ x, const W* __restrict__ gamma,
                            uint8_t* __restrict__ q, float* __restrict__ scale,
                            float* __restrict__ rstd, int64_t M, int N, float eps, int gemma) {
  using E = Elem<T>;
  __shared__ float red_s[8], red_m[8];
  const int64_t row = blockIdx.x;
  const T* xr = x + row * N;
  pdl_trigger();
  pdl_wait();
  Kahan1 acc;
  for (int j = threadIdx.x; j < N; j += 256) {
    const float f = E::to_f(xr[j]);
    acc.add(__fmul_rn(f, f));
  }
  const float ss = group_sum(acc.total(), 256, 0, red_s);
  const float r = 1.0f / sqrtf(ss / (float)N + eps);
  auto y_at = [&](int j) {
    const float f = E::to_f(xr[j]);
    const float g = Elem<W>::to_f(gamma[j]);
    const float o = gemma ? (f * r) * (1.0f + g) : Elem<W>::round(f * r) * g;
    return E::to_f(E::from_f(o));  // the stored value
  };
  float am = 0.f;
  for (int j = threadIdx.x; j < N; j += 256) am = fmaxf(am, fabsf(y_at(j)));
  const float amax = group_max(am, 256, 0, red_m);
  const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 1.0f;
  if (threadIdx.x == 0) {
    rstd[row] = r;
    scale[row] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  }
  uint8_t* qr = q + row * (int64_t)N;
  for (int j = threadIdx.x; j < N; j += 256)
    qr[j] = (uint8_t)(f2_to_e4m3x2(__fmul_rn(y_at(j), inv), 0.f) & 0xffu);
}

// Aligned rows too wide for registers (any width): one CTA of 1024 threads
// per row walks the row in 16-byte vectors three times: the sum of squares;
// y as the forward stores it and its absolute maximum; y again (the same
// instructions, so the same values) and the codes.  The first pass brings
// the row from HBM; the later passes find it in L2 (a CTA's row is at most
// a few hundred KiB, and one or two rows per SM are in flight).  A thread
// adds up to N/8192 vectors in sequence, so each vector's partial enters a
// compensated sum.  kLoads vectors per thread are in flight per step.
constexpr int kQuantLoopThreads = 1024;

template <typename T, typename W, bool GEMMA>
__global__ void __launch_bounds__(kQuantLoopThreads)
rms_fwd_quant_looped_kernel(const T* __restrict__ x, const W* __restrict__ gamma,
                            uint8_t* __restrict__ q, float* __restrict__ scale,
                            float* __restrict__ rstd, int N, float eps) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  constexpr int NP = Pairs<T>::n;
  constexpr int kLoads = 4;
  constexpr int kStep = kLoads * kQuantLoopThreads;
  __shared__ float red_s[32], red_m[32];
  const int NV = N / VN;
  const int64_t row = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x) + row * (int64_t)NV;
  pdl_trigger();
  pdl_wait();

  Kahan1 acc;
  for (int v0 = threadIdx.x; v0 < NV; v0 += kStep) {
    uint4 t[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int v = v0 + u * kQuantLoopThreads;
      t[u] = v < NV ? ld_keep(xr + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      f32x2 ss2 = 0ull;
      Math::sumsq(t[u], ss2);
      acc.add(lo2(ss2) + hi2(ss2));
    }
  }
  const float ss = group_sum(acc.total(), kQuantLoopThreads, 0, red_s);
  const float r = 1.0f / sqrtf(ss / (float)N + eps);

  AbsMax<T> am;
  for (int v0 = threadIdx.x; v0 < NV; v0 += kStep) {
    uint4 t[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int v = v0 + u * kQuantLoopThreads;
      t[u] = v < NV ? ld_keep(xr + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int v = v0 + u * kQuantLoopThreads;
      if (v < NV) am.add(Math::forward(t[u], GV::load(gamma, v), r));
    }
  }
  const float amax = group_max(am.value(), kQuantLoopThreads, 0, red_m);
  const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 1.0f;
  if (threadIdx.x == 0) {
    rstd[row] = r;
    scale[row] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  }

  uint8_t* qr = q + row * (int64_t)N;
  const f32x2 iv = splat2(inv);
  for (int v0 = threadIdx.x; v0 < NV; v0 += kStep) {
    uint4 t[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int v = v0 + u * kQuantLoopThreads;
      t[u] = v < NV ? ld_stream(xr + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int v = v0 + u * kQuantLoopThreads;
      if (v < NV) {
        const uint4 yv = Math::forward(t[u], GV::load(gamma, v), r);
        uint32_t c[NP];
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          const f32x2 p = mul2(stored_pair<T>(yv, i), iv);
          c[i] = f2_to_e4m3x2(lo2(p), hi2(p));
        }
        if constexpr (NP == 4) {
          *reinterpret_cast<uint2*>(qr + (int64_t)v * VN) =
              make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
        } else {
          *reinterpret_cast<uint32_t*>(qr + (int64_t)v * VN) = c[0] | (c[1] << 16);
        }
      }
    }
  }
}

template <typename F>
cudaError_t quant_types(int dtype, int gemma, F&& f) {
  auto g = [&](auto* tp, auto* wp) -> cudaError_t {
    return gemma ? f(tp, wp, std::true_type{}) : f(tp, wp, std::false_type{});
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

// Rows of up to 32 KiB in registers.  Rows of more than 512 vectors take
// eight vectors a thread (rms_fwd_quant_pairs_kernel: a thread for every
// two of the register forward's Gv threads), so the per-row work of this
// kernel (two group reductions, the square root, the scale's division) is
// spread over twice the data.  m.kv = 8 marks it; m.sv carries Gv.
// Measured on GB300: 16384 x 8192 bf16 74.1 -> 70.9 us; at 8192 x 4096 the
// register forward's four vectors a thread stay faster (21.3 against
// 22.3 us), so narrower rows keep its plan.
#ifndef RMS_QUANT_KV8_MIN_NV
#define RMS_QUANT_KV8_MIN_NV 513
#endif
// CTAs of at least this many threads (several rows a CTA when a row has
// fewer): GB300, 8192 x 4096 bf16 with one 128-thread row a CTA 20.4 us
// against 21.2 us with two rows in 256-thread CTAs (512: 23.0 us).
#ifndef RMS_QUANT_MIN_CTA_THREADS
#define RMS_QUANT_MIN_CTA_THREADS 128
#endif
#ifndef RMS_QUANT_NARROW_KV4
#define RMS_QUANT_NARROW_KV4 1
#endif
bool plan_quant_registers(int N, int dtype, Mapping* m) {
  if (!plan_registers(N, dtype, false, m)) return false;
  if (m->threads > 512) return false;
  const int NV = (int)(((int64_t)N * dtype_bytes(dtype)) / 16);
  if (NV <= 128 && RMS_QUANT_NARROW_KV4) {
    // Rows of up to 128 vectors: four vectors a lane, a power-of-two group
    // of lanes a row (several rows a warp), so the per-row work (the two
    // reductions, the square root, the divisions) is spread over four
    // vectors a thread instead of one or two.
    int G = 1;
    while (4 * G < NV) G *= 2;
    m->kv = 4;
    m->G = G;
  }
  if (m->G < 256) {
    m->rows_per_cta = m->G >= RMS_QUANT_MIN_CTA_THREADS ? 1 : RMS_QUANT_MIN_CTA_THREADS / m->G;
    m->threads = m->G * m->rows_per_cta;
  }
  if (NV < RMS_QUANT_KV8_MIN_NV || NV <= 128) return true;
  const int Gv = m->G;  // >= 64: four vectors a thread, NV > 128
  const int G = (Gv / 2 + 31) / 32 * 32;
  m->kv = 8;
  m->sv = Gv;
  m->G = G;
  m->rows_per_cta = G >= RMS_QUANT_MIN_CTA_THREADS ? 1 : RMS_QUANT_MIN_CTA_THREADS / G;
  m->threads = G * m->rows_per_cta;
  return true;
}

cudaError_t launch_fwd_quant(const QuantArgs& a, const Mapping& m, cudaStream_t s) {
  return rmsk::quant_types(a.dtype, a.gemma, [&](auto* tp, auto* wp, auto gm) -> cudaError_t {
    using T = std::remove_pointer_t<decltype(tp)>;
    using W = std::remove_pointer_t<decltype(wp)>;
    constexpr bool GEMMA = decltype(gm)::value;
    const T* x = static_cast<const T*>(a.x);
    const W* g = static_cast<const W*>(a.gamma);
    if (m.path == kRegisters) {
      const dim3 grid((unsigned)((a.M + m.rows_per_cta - 1) / m.rows_per_cta)), block(m.threads);
      switch (m.kv) {
        case 1: return rmsk::launch_pdl(rmsk::rms_fwd_quant_registers_kernel<T, W, 1, GEMMA>, grid, block, 0, s, x, g, a.q, a.scale, a.rstd, a.M, a.N, a.eps, m.G);
        case 2: return rmsk::launch_pdl(rmsk::rms_fwd_quant_registers_kernel<T, W, 2, GEMMA>, grid, block, 0, s, x, g, a.q, a.scale, a.rstd, a.M, a.N, a.eps, m.G);
        case 8: return rmsk::launch_pdl(rmsk::rms_fwd_quant_pairs_kernel<T, W, GEMMA>, grid, block, 0, s, x, g, a.q, a.scale, a.rstd, a.M, a.N, a.eps, m.G, m.sv);
        default: return rmsk::launch_pdl(rmsk::rms_fwd_quant_registers_kernel<T, W, 4, GEMMA>, grid, block, 0, s, x, g, a.q, a.scale, a.rstd, a.M, a.N, a.eps, m.G);
      }
    }
    if (m.path == kChunked)
      return rmsk::launch_pdl(rmsk::rms_fwd_quant_looped_kernel<T, W, GEMMA>, dim3((unsigned)a.M),
                              dim3(rmsk::kQuantLoopThreads), 0, s, x, g, a.q, a.scale, a.rstd,
                              a.N, a.eps);
    return rmsk::launch_pdl(rmsk::rms_fwd_quant_scalar_kernel<T, W>, dim3((unsigned)a.M), dim3(256),
                            0, s, x, g, a.q, a.scale, a.rstd, a.M, a.N, a.eps, a.gemma);
  });
}

}  // namespace rmsi
