// Forward RMSNorm, register mapping: a group of G threads (one warp, or
// several warps up to the whole CTA) owns one row and holds it in registers
// as 16-byte vectors, so x is read from HBM exactly once and y written once.
//
//   r = 1 / sqrt(sum(x^2) / N + eps)        (the true N, never a padded width)
//   y = round(round(x * r) * gamma)         (non-Gemma: normalised row cast to
//                                            the weight dtype, then weighted)
//   y = round(x * r * (1 + gamma))          (Gemma)
//
// Sources: "Hướng dẫn Triton RMSNorm: kernel, backward…", sections "Vấn đề
// và công thức tham chiếu" and "N và BLOCK: hai kích thước không được nhầm";
// "02 · 手写 Triton kernel:RMSNorm / RoPE / SwiGLU", section 3 (cast order,
// Gemma weight).
#include "common.cuh"
#include "internal.h"

namespace rmsk {

// With RES the row normalised is h = x + residual (rounded to T), which is
// also stored to h (h may be the residual buffer itself: each thread reads
// its residual vectors before it overwrites them).
template <typename T, typename W, int KV, bool GEMMA, bool RES>
__global__ void __launch_bounds__(RES ? 512 : 1024)
rms_fwd_registers_kernel(const T* __restrict__ x, const W* __restrict__ gamma, T* __restrict__ y,
                         float* __restrict__ rstd, int64_t M, int N, float eps, int G,
                         const T* res, T* h) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  __shared__ float red[32];
  const int NV = N / VN;
  const int grp = threadIdx.x / G;
  const int lig = threadIdx.x - grp * G;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / G) + grp;
  const bool active = row < M;
  const int64_t base = (active ? row : 0) * (int64_t)NV;
  const uint4* xr = reinterpret_cast<const uint4*>(x) + base;
  pdl_trigger();
  pdl_wait();

  uint4 xv[KV], rv[RES ? KV : 1];
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = lig + k * G;
    const bool in = active && v < NV;
    xv[k] = in ? ld_stream(xr + v) : make_uint4(0u, 0u, 0u, 0u);
    if (RES) rv[k] = in ? ld_stream(reinterpret_cast<const uint4*>(res) + base + v)
                        : make_uint4(0u, 0u, 0u, 0u);
  }
  if (RES) {
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = lig + k * G;
      xv[k] = Math::add_round(xv[k], rv[k]);  // zero vectors stay zero
      if (active && v < NV) st_stream(reinterpret_cast<uint4*>(h) + base + v, xv[k]);
    }
  }
  f32x2 ss2 = 0ull;
#pragma unroll
  for (int k = 0; k < KV; ++k) Math::sumsq(xv[k], ss2);
  // Rows of at most 16 vectors (KV = 1) may give each row a sub-warp group.
  const float ss = (KV == 1 && G < 32) ? lane_group_sum(lo2(ss2) + hi2(ss2), G)
                                       : group_sum(lo2(ss2) + hi2(ss2), G, grp * (G >> 5), red);
  const float r = 1.0f / sqrtf(ss / (float)N + eps);
  if (!active) return;  // no barrier follows
  if (lig == 0) rstd[row] = r;

  uint4* yr = reinterpret_cast<uint4*>(y) + row * (int64_t)NV;
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = lig + k * G;
    if (v < NV) st_stream(yr + v, Math::forward(xv[k], GV::load(gamma, v), r));
  }
}

template <typename T, typename W, bool GEMMA, bool RES>
static cudaError_t launch_g(const rmsi::FwdArgs& a, const rmsi::Mapping& m, cudaStream_t s) {
  const dim3 grid((unsigned)m.blocks), block(m.threads);
  const T* x = static_cast<const T*>(a.x);
  const W* g = static_cast<const W*>(a.gamma);
  T* y = static_cast<T*>(a.y);
  const T* r = static_cast<const T*>(a.res);
  T* h = static_cast<T*>(a.h);
  switch (m.kv) {
    case 1: return launch_pdl(rms_fwd_registers_kernel<T, W, 1, GEMMA, RES>, grid, block, 0, s, x, g, y, a.rstd, a.M, a.N, a.eps, m.G, r, h);
    case 2: return launch_pdl(rms_fwd_registers_kernel<T, W, 2, GEMMA, RES>, grid, block, 0, s, x, g, y, a.rstd, a.M, a.N, a.eps, m.G, r, h);
    case 4: return launch_pdl(rms_fwd_registers_kernel<T, W, 4, GEMMA, RES>, grid, block, 0, s, x, g, y, a.rstd, a.M, a.N, a.eps, m.G, r, h);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, typename W>
static cudaError_t launch_t(const rmsi::FwdArgs& a, const rmsi::Mapping& m, cudaStream_t s) {
  if (a.res) return a.gemma ? launch_g<T, W, true, true>(a, m, s) : launch_g<T, W, false, true>(a, m, s);
  return a.gemma ? launch_g<T, W, true, false>(a, m, s) : launch_g<T, W, false, false>(a, m, s);
}

}  // namespace rmsk

namespace rmsi {

// Threads per row and vectors per thread for a row of N elements held in
// registers.  Rows of up to 16 vectors get a power-of-two group of lanes
// (several rows per warp); rows of up to 128 vectors (2 KiB) one warp each,
// several rows per CTA; wider rows ceil(vectors / 4) threads rounded up to a
// warp multiple, up to 1024 threads (wider rows use the staged mapping).
bool plan_registers(int N, int dtype, bool bwd, Mapping* m) {
  const int b = dtype_bytes(dtype);
  if (N <= 0 || ((int64_t)N * b) % 16 != 0) return false;
  const int NV = (int)(((int64_t)N * b) / 16);
  const int max_threads = bwd ? 512 : 1024;
  int kv, G;
  if (NV <= 16) {
    // Narrow rows: a power-of-two group of lanes per row, several rows per
    // warp, so no lane idles beyond the rounding of NV up to a power of two.
    kv = 1;
    G = 1;
    while (G < NV) G *= 2;
  } else if (NV <= 32) {
    kv = 1; G = 32;
  } else if (NV <= 64) {
    kv = 2; G = 32;
  } else if (NV <= 128) {
    kv = 4; G = 32;
  } else {
    kv = 4;
    G = ((NV + 3) / 4 + 31) / 32 * 32;
    if (G > max_threads) return false;
  }
  m->path = kRegisters;
  m->kv = kv;
  m->G = G;
  // A row of two to four warps is a CTA of its own (GB300 forward: 8192 x
  // 4096 bf16 23.1 -> 21.9 us, 32768 x 3072 Gemma 64.0 -> 61.2 us against two
  // rows in 256-thread CTAs); rows of a warp or less share 256-thread CTAs.
  m->rows_per_cta = G >= 64 ? (G >= 128 ? 1 : 128 / G) : 256 / G;
  m->threads = G * m->rows_per_cta;
  m->smem = 0;
  return true;
}

cudaError_t launch_fwd_registers(const FwdArgs& a, const Mapping& m0, cudaStream_t s) {
  Mapping m = m0;
  m.blocks = (a.M + m.rows_per_cta - 1) / m.rows_per_cta;
  switch (a.dtype) {
    case kBF16: return rmsk::launch_t<__nv_bfloat16, __nv_bfloat16>(a, m, s);
    case kF16: return rmsk::launch_t<__half, __half>(a, m, s);
    case kBF16W32: return rmsk::launch_t<__nv_bfloat16, float>(a, m, s);
    case kF16W32: return rmsk::launch_t<__half, float>(a, m, s);
    default: return rmsk::launch_t<float, float>(a, m, s);
  }
}

}  // namespace rmsi
