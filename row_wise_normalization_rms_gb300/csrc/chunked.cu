// RMSNorm for rows wider than one CTA holds: the row is never held on chip
// whole, so every pass streams it from memory.
//
// One-pass mapping (rows up to 16 slices): a thread-block cluster of C CTAs
// takes each row, CTA rank c the column slice [c*SV, (c+1)*SV).  First pass:
// the slice comes from HBM into registers and the CTA's partial sum goes to
// every CTA of the cluster (st.async into a slot of its shared memory,
// completing on its mbarrier); while those arrive, the slice of the
// cluster's next row is already on its way.  Second pass: every CTA adds the
// C partials in rank order (the same total in each) and writes the outputs
// -- the backward from the slice it held in registers, the forward from the
// slice read again from L2, where the first pass left it a moment before.
// HBM sees every input once.  The backward keeps dgamma partials of its
// slice in registers across the cluster's rows; the fixed-order column
// reduction finishes dgamma.
//
// Three-pass mapping (wider rows): a row pass computes r (forward) or
// k = r * mean(u * x) (backward) per row, then (row, chunk) units write the
// outputs, re-reading the row from memory; no width limit.
//
// Sources: "Hướng dẫn Triton RMSNorm: kernel, backward…", sections "Vấn đề
// và công thức tham chiếu" (r, y) and "Backward đầu vào: giữ đúng N" (dx,
// dgamma); the looped row reduction for rows wider than one block is the
// LN chapter's ("第 07 章:LayerNorm——反向传播与原子锁", step 3).
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "e4m3.cuh"
#include "internal.h"
#include "tma.cuh"

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

// Row pass of the three-pass mapping.  Forward: out = r = 1/sqrt(sum(x^2)/N
// + eps); with RES the row is h = x + res, stored to h for the normalise
// pass.  Backward: out = k = sum(u * x * r)/N.  C CTAs share a row (C > 1:
// a thread-block cluster, CTA rank c taking vectors [c*SV, (c+1)*SV)), so a
// few rows still fill the GPU; their sums meet in rank order through
// distributed shared memory after one cluster barrier per row (slots
// alternate, so one barrier suffices).  Rows are grid-strided by cluster.
template <typename T, typename W, bool GEMMA, bool BWD, bool RES>
__global__ void __launch_bounds__(kChunkThreads)
rms_rowstat_kernel(const T* __restrict__ x, const T* __restrict__ dy, const W* __restrict__ gamma,
                   const float* __restrict__ rstd_in, float* __restrict__ out, int64_t M, int N,
                   float eps, const T* res, T* h, int C, int SV) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  __shared__ float red[2 * 32];
  __shared__ float slot[2];
  const int NV = N / VN;
  const int rank = C > 1 ? (int)cluster_rank() : 0;
  const int vbeg = rank * SV;
  const int vend = min(NV, vbeg + SV);
  pdl_wait();
  int buf = 0;
  for (int64_t row = blockIdx.x / C; row < M; row += gridDim.x / C, buf ^= 1) {
    const uint4* xr = reinterpret_cast<const uint4*>(x) + row * (int64_t)NV;
    const uint4* dr = reinterpret_cast<const uint4*>(dy) + row * (int64_t)NV;
    const float r = BWD ? rstd_in[row] : 0.f;
    Kahan2 acc;  // a thread adds (vend - vbeg) / kChunkSpan partial sums in sequence
    for (int v0 = vbeg + (int)threadIdx.x; v0 < vend; v0 += kChunkSpan) {
      uint4 xv[kChunkVecs], dv[kChunkVecs];
#pragma unroll
      for (int u = 0; u < kChunkVecs; ++u) {
        const int v = v0 + u * kChunkThreads;
        xv[u] = v < vend ? ld_keep(xr + v) : make_uint4(0u, 0u, 0u, 0u);
        if (BWD || RES) {
          const uint4* src = BWD ? dr : reinterpret_cast<const uint4*>(res) + row * (int64_t)NV;
          dv[u] = v < vend ? ld_stream(src + v) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (RES) {
#pragma unroll
        for (int u = 0; u < kChunkVecs; ++u) {
          const int v = v0 + u * kChunkThreads;
          xv[u] = Math::add_round(xv[u], dv[u]);
          if (v < vend) __stcg(reinterpret_cast<uint4*>(h) + row * (int64_t)NV + v, xv[u]);
        }
      }
      f32x2 part = 0ull;
#pragma unroll
      for (int u = 0; u < kChunkVecs; ++u) {
        const int v = v0 + u * kChunkThreads;
        if (v < vend) {
          if (BWD) {
            Math::backward_dot(xv[u], dv[u], GV::load(gamma, v), r, part);
          } else {
            Math::sumsq(xv[u], part);
          }
        }
      }
      acc.add(part);
    }
    float tot = cta_sum(acc.total(), red, buf);
    if (C > 1) {
      if (threadIdx.x == 0) slot[buf] = tot;
      cluster_sync();
      if (rank == 0 && threadIdx.x == 0) {
        const uint32_t a = smem_u32(&slot[buf]);
        tot = 0.f;
        for (int c = 0; c < C; ++c) tot += ld_cluster_f32(map_to_rank(a, (uint32_t)c));
      }
    }
    if (rank == 0 && threadIdx.x == 0)
      out[row] = BWD ? tot / (float)N : 1.0f / sqrtf(tot / (float)N + eps);
  }
  if (C > 1) cluster_sync();  // rank 0 may still be reading this CTA's slot
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


// ---- one-pass mapping: a cluster of CTAs per row ------------------------------
constexpr int kWideThreads = 512;
constexpr int kWideWarps = kWideThreads / 32;
constexpr int kWideMaxCluster = 16;            // non-portable cluster size
constexpr int kWideGammaSmem = 128 * 1024;     // the CTA's weight slice in shared memory

struct WideParams {
  const void* x;
  const void* gamma;
  const void* in2;  // backward: dy; fused forward: the residual
  const void* in3;  // fused backward: dh
  void* out;        // forward: y; backward: dx (may equal dy, or dh)
  void* h;          // fused forward: h = x + residual (may equal the residual)
  float* rstd;      // forward: written; backward: read
  float* ws;        // backward: [units][N] column partials
  int64_t M;
  int N;
  float eps;
  int C;   // CTAs per cluster
  int SV;  // 16-byte vectors per CTA slice: KV * kWideThreads
  long long wait_limit;  // polls of an exchange wait before the status word is raised
};

// Nonzero once an exchange wait of a one-pass kernel ran past the wait
// limit; read and cleared by the host.
__device__ int g_wide_device_status = 0;

// Row-partial exchange of the one-pass kernels.  Slot [buf][c] of every CTA
// of the cluster receives CTA c's partial of the row: from each peer by
// st.async, which completes 4 transaction bytes on the receiver's barrier
// bars[buf]; its own by a plain store followed by this CTA's one arrival on
// bars[buf], which also expects the (C-1)*4 bytes of the peers.  No fence
// and no cluster barrier per row.  Rows alternate between the two
// slots/barriers (buf); a CTA pushes row i only after completing row i-1,
// which needed the receiver's push of row i-1, made after the receiver had
// finished with row i-2: so a push of row i never meets slot or barrier
// state of row i-2.  With C == 1 no cluster instruction is used.
struct WideExchange {
  uint64_t bars[2];
  float slots[2][kWideMaxCluster];
};

__device__ __forceinline__ void wide_init(WideExchange& x, int C) {
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&x.bars[0]), 1);
    mbar_init(smem_u32(&x.bars[1]), 1);
    fence_mbar_init();
  }
  if (C > 1) {
    cluster_sync();  // every CTA's barriers exist before any push
  } else {
    __syncthreads();
  }
}

// This CTA's sum of one float per thread (warps in order), or with MAX its
// maximum: thread c sends it to slot [buf][rank] of CTA c (thread `rank`
// writes its own CTA's slot and arrives).  `red` alternates with buf, so the
// one CTA barrier here suffices.
template <bool MAX = false, int NW = kWideWarps>
__device__ __forceinline__ void wide_publish(float v, float (*red)[NW], WideExchange& x,
                                             int buf, int rank, int C) {
  if (MAX) {
    asm volatile("redux.sync.max.f32 %0, %0, 0xffffffff;" : "+f"(v));  // as fmaxf over the warp
  } else {
    v = warp_sum(v);
  }
  if ((threadIdx.x & 31) == 0) red[buf][threadIdx.x >> 5] = v;
  __syncthreads();
  if ((int)threadIdx.x < C) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) t = MAX ? fmaxf(t, red[buf][w]) : t + red[buf][w];
    const uint32_t bar = smem_u32(&x.bars[buf]);
    if ((int)threadIdx.x == rank) {
      x.slots[buf][rank] = t;
      // The arrival releases the slot store to the CTA's waiting threads.
      if (C == 1) {
        mbar_arrive(bar);
      } else {
        mbar_arrive_expect_tx(bar, 4u * (uint32_t)(C - 1));
      }
    } else {
      const uint32_t slot = smem_u32(&x.slots[buf][rank]);
      st_async_f32(map_to_rank(slot, threadIdx.x), t, map_to_rank(bar, threadIdx.x));
    }
  }
}

// The row total once all C partials of slot `buf` are in (barrier phase
// parity `parity`): the slots in rank order.  A wait that runs past `limit`
// polls raises the status word and then waits out the phase (bounded): the
// exchange never skips a row, so every CTA keeps the same barrier phases.
// With MAX the slots' maximum (order-free).
template <bool MAX = false>
__device__ __forceinline__ float wide_total(WideExchange& x, int buf, uint32_t parity, int C,
                                            long long limit) {
  const uint32_t bar = smem_u32(&x.bars[buf]);
  if (!mbar_wait(bar, parity, limit)) {
    g_wide_device_status = 1;
    mbar_wait(bar, parity, kDrainPolls);
  }
  float t = 0.f;
  for (int c = 0; c < C; ++c) t = MAX ? fmaxf(t, x.slots[buf][c]) : t + x.slots[buf][c];
  return t;
}

// Forward.  Thread t owns vectors v0 + t + k*kWideThreads (k < KV) of every
// row of its cluster; rows u, u + U, ... for cluster u of U.  The slice of
// the next row is loaded while the current one is exchanged; the second
// pass reads the current slice again, from L2 (holding it in registers
// instead costs the second CTA per SM, and measured slower on GB300).  With
// RES the first pass forms h = x + residual, stores it and reduces it.
template <typename T, typename W, int KV, bool GEMMA, bool RES>
__global__ void __launch_bounds__(kWideThreads, KV <= 4 ? 2 : 1)
rms_fwd_wide_kernel(const WideParams p) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  extern __shared__ __align__(16) uint8_t wide_smem[];
  GV* gs = reinterpret_cast<GV*>(wide_smem);  // this thread's weights at [t + k*kWideThreads]
  __shared__ float red[2][kWideWarps];
  __shared__ WideExchange xch;
  const int NV = p.N / VN;
  const int rank = p.C > 1 ? (int)cluster_rank() : 0;
  const int64_t unit = blockIdx.x / p.C;
  const int64_t units = gridDim.x / p.C;
  const int tid = threadIdx.x;
  const int v0 = rank * p.SV + tid;
  wide_init(xch, p.C);
  pdl_wait();
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = v0 + k * kWideThreads;
    if (v < NV) gs[tid + k * kWideThreads] = GV::load(p.gamma, v);
  }

  uint4 a[KV], b[RES ? KV : 1];  // the slice of the next row, as loaded
  auto fetch = [&](int64_t row) {
    const uint4* xr = static_cast<const uint4*>(p.x) + row * (int64_t)NV;
    const uint4* rr = static_cast<const uint4*>(p.in2) + row * (int64_t)NV;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = v0 + k * kWideThreads;
      a[k] = v < NV ? __ldcg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
      if (RES) b[k] = v < NV ? __ldcg(rr + v) : make_uint4(0u, 0u, 0u, 0u);
    }
  };

  int64_t row = unit;
  if (row < p.M) fetch(row);
  for (int it = 0; row < p.M; ++it) {
    const int buf = it & 1;
    // First pass: the slice's sum of squares.
    Kahan2 ss;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = v0 + k * kWideThreads;
      uint4 hv = a[k];
      if (v < NV) {
        if (RES) {
          hv = Math::add_round(a[k], b[k]);
          __stcg(static_cast<uint4*>(p.h) + row * (int64_t)NV + v, hv);
        }
        f32x2 t = 0ull;
        Math::sumsq(hv, t);
        ss.add(t);
      }
    }
    wide_publish(ss.total(), red, xch, buf, rank, p.C);
    const int64_t next = row + units;
    if (next < p.M) fetch(next);  // in flight across the exchange and the second pass
    const float tot = wide_total(xch, buf, (uint32_t)(it >> 1) & 1u, p.C, p.wait_limit);
    const float r = 1.0f / sqrtf(tot / (float)p.N + p.eps);
    if (rank == 0 && tid == 0) p.rstd[row] = r;
    // Second pass: the slice again, now from L2.
    const uint4* src = static_cast<const uint4*>(RES ? p.h : p.x) + row * (int64_t)NV;
    uint4* yr = static_cast<uint4*>(p.out) + row * (int64_t)NV;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = v0 + k * kWideThreads;
      if (v < NV) {
        st_stream(yr + v, Math::forward(__ldcs(src + v), gs[tid + k * kWideThreads], r));
      }
    }
    row = next;
  }
  if (p.C > 1) cluster_sync();
}

// Forward with an FP8 E4M3 output for rows a CTA cannot hold in registers:
// the cluster mapping of rms_fwd_wide_kernel (KV = 4; CTAs of TPB threads,
// 1024 / TPB of them an SM at least), with
// two exchanges per row instead of one: the slice's sum of squares (giving
// r), then the slice's maximum of |y| (giving the row's scale).  HBM is read
// once: each thread keeps its vectors of the current row in shared memory
// (its own slots, so no barrier) while its registers take the next row's;
// the pass that finds the maximum replaces them there by y, which the last
// pass turns into codes.  The exchanges of a row are consecutive steps of the one slot
// sequence (step k uses slot and barrier k & 1), so the ordering argument of
// WideExchange holds step by step.  q is p.out, the per-row scale p.h.
template <typename T, typename W, bool GEMMA, int TPB>
__global__ void __launch_bounds__(TPB, 1024 / TPB)
rms_fwd_quant_wide_kernel(const WideParams p) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  constexpr int KV = 4;
  constexpr int VN = Elem<T>::kPerVec;
  constexpr int NP = Pairs<T>::n;
  extern __shared__ __align__(16) uint8_t wide_smem[];
  GV* gs = reinterpret_cast<GV*>(wide_smem);  // this thread's weights at [t + k*TPB]
  uint4* xs = reinterpret_cast<uint4*>(wide_smem + (size_t)p.SV * sizeof(GV));  // the row's slice
  __shared__ float red[2][TPB / 32];
  __shared__ WideExchange xch;
  uint8_t* q = static_cast<uint8_t*>(p.out);
  float* scale = static_cast<float*>(p.h);
  const int NV = p.N / VN;
  const int rank = p.C > 1 ? (int)cluster_rank() : 0;
  const int64_t unit = blockIdx.x / p.C;
  const int64_t units = gridDim.x / p.C;
  const int tid = threadIdx.x;
  const int v0 = rank * p.SV + tid;
  wide_init(xch, p.C);
  pdl_wait();
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = v0 + k * TPB;
    if (v < NV) gs[tid + k * TPB] = GV::load(p.gamma, v);
  }

  uint4 a[KV];  // the slice of the next row, as loaded
  auto fetch = [&](int64_t row) {
    const uint4* xr = static_cast<const uint4*>(p.x) + row * (int64_t)NV;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = v0 + k * TPB;
      a[k] = v < NV ? __ldcg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
    }
  };

  int64_t row = unit;
  if (row < p.M) fetch(row);
  uint32_t step = 0;  // exchanges so far
  while (row < p.M) {
    // First pass: the slice's sum of squares (a thread's four vectors in one
    // chain per lane, as the register mappings add at most 32 terms a
    // thread); the slice kept on chip.
    float ss_lo = 0.f, ss_hi = 0.f;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      if (v0 + k * TPB < NV) {
        SumSqDirect<T>::add(a[k], ss_lo, ss_hi);
        xs[tid + k * TPB] = a[k];
      }
    }
    wide_publish<false, TPB / 32>(ss_lo + ss_hi, red, xch, (int)(step & 1), rank, p.C);
    const int64_t next = row + units;
    if (next < p.M) fetch(next);  // in flight across both exchanges
    const float tot = wide_total(xch, (int)(step & 1), (step >> 1) & 1u, p.C, p.wait_limit);
    ++step;
    const float r = 1.0f / sqrtf(tot / (float)p.N + p.eps);
    // Second pass: y (kept on chip in place of the slice) and its largest
    // magnitude.
    AbsMax<T> am;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int i = tid + k * TPB;
      if (v0 + k * TPB < NV) {
        const uint4 yv = Math::forward(xs[i], gs[i], r);
        xs[i] = yv;
        am.add(yv);
      }
    }
    wide_publish<true, TPB / 32>(am.value(), red, xch, (int)(step & 1), rank, p.C);
    const float amax = wide_total<true>(xch, (int)(step & 1), (step >> 1) & 1u, p.C, p.wait_limit);
    ++step;
    const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 1.0f;
    if (rank == 0 && tid == 0) {
      p.rstd[row] = r;
      scale[row] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    }
    // Third pass: the codes of the held y.
    uint8_t* qr = q + row * (int64_t)p.N;
    const f32x2 iv = splat2(inv);
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = v0 + k * TPB;
      if (v < NV) {
        const uint4 yv = xs[tid + k * TPB];
        uint32_t c[NP];
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          const f32x2 pr = mul2(stored_pair<T>(yv, i), iv);
          c[i] = f2_to_e4m3x2(lo2(pr), hi2(pr));
        }
        if constexpr (NP == 4) {
          __stcs(reinterpret_cast<uint2*>(qr + (int64_t)v * VN),
                 make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16)));
        } else {
          __stcs(reinterpret_cast<unsigned int*>(qr + (int64_t)v * VN), c[0] | (c[1] << 16));
        }
      }
    }
    row = next;
  }
  if (p.C > 1) cluster_sync();
}

// Backward (KV = 4, one CTA per SM): first pass r*sum(u*x) over the slice;
// second pass dgamma terms and dx (+ dh with RES) from the held slice while
// the next row's slice loads.  The cluster's dgamma partial for its slice
// goes to workspace row u.
template <typename T, typename W, bool GEMMA, bool RES>
__global__ void __launch_bounds__(kWideThreads, 1)
rms_bwd_wide_kernel(const WideParams p) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  constexpr int NP = Math::kPairs;
  constexpr int KV = 4;
  extern __shared__ __align__(16) uint8_t wide_smem[];
  GV* gs = reinterpret_cast<GV*>(wide_smem);
  __shared__ float red[2][kWideWarps];
  __shared__ WideExchange xch;
  const int NV = p.N / VN;
  const int rank = p.C > 1 ? (int)cluster_rank() : 0;
  const int64_t unit = blockIdx.x / p.C;
  const int64_t units = gridDim.x / p.C;
  const int tid = threadIdx.x;
  const int v0 = rank * p.SV + tid;
  wide_init(xch, p.C);
  pdl_wait();
  f32x2 acc[KV][NP];
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = v0 + k * kWideThreads;
    if (v < NV) gs[tid + k * kWideThreads] = GV::load(p.gamma, v);
#pragma unroll
    for (int e = 0; e < NP; ++e) acc[k][e] = 0ull;
  }

  uint4 a[KV], d[KV];      // the next row's slice, as loaded
  uint4 xc[KV], dc[KV];    // the current row's slice
  float r_next = 0.f;
  auto fetch = [&](int64_t row) {
    const uint4* xr = static_cast<const uint4*>(p.x) + row * (int64_t)NV;
    const uint4* dr = static_cast<const uint4*>(p.in2) + row * (int64_t)NV;
    r_next = p.rstd[row];
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = v0 + k * kWideThreads;
      a[k] = v < NV ? __ldcg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
      d[k] = v < NV ? __ldcg(dr + v) : make_uint4(0u, 0u, 0u, 0u);
    }
  };

  int64_t row = unit;
  if (row < p.M) fetch(row);
  for (int it = 0; row < p.M; ++it) {
    const int buf = it & 1;
    const float r = r_next;
    Kahan2 sux;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = v0 + k * kWideThreads;
      xc[k] = a[k];
      dc[k] = d[k];
      if (v < NV) {
        f32x2 t = 0ull;
        Math::backward_dot(xc[k], dc[k], gs[tid + k * kWideThreads], r, t);
        sux.add(t);
      }
    }
    wide_publish(sux.total(), red, xch, buf, rank, p.C);
    const int64_t next = row + units;
    if (next < p.M) fetch(next);
    const float tot = wide_total(xch, buf, (uint32_t)(it >> 1) & 1u, p.C, p.wait_limit);
    const float kc = tot / (float)p.N;  // r * mean(u*x)
    uint4* out = static_cast<uint4*>(p.out) + row * (int64_t)NV;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = v0 + k * kWideThreads;
      if (v < NV) {
        const GV g = gs[tid + k * kWideThreads];
        Math::backward_acc(xc[k], dc[k], r, acc[k]);
        if constexpr (RES) {
          const uint4 hv = __ldcs(static_cast<const uint4*>(p.in3) + row * (int64_t)NV + v);
          st_stream(out + v, Math::backward_dx_add(xc[k], dc[k], g, r, kc, hv));
        } else {
          st_stream(out + v, Math::backward_dx(xc[k], dc[k], g, r, kc));
        }
      }
    }
    row = next;
  }
  float* wp = p.ws + unit * (int64_t)p.N;
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = v0 + k * kWideThreads;
    if (v < NV) {
      float4* w4 = reinterpret_cast<float4*>(wp + (int64_t)v * VN);
#pragma unroll
      for (int q = 0; q < NP / 2; ++q)
        w4[q] = make_float4(lo2(acc[k][2 * q]), hi2(acc[k][2 * q]), lo2(acc[k][2 * q + 1]),
                            hi2(acc[k][2 * q + 1]));
    }
  }
  if (p.C > 1) cluster_sync();
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

// Vectors per thread of the one-pass mapping (the slice of a CTA is KV *
// 512 vectors), or 0 when its slices would need more than kWideMaxCluster
// CTAs.  Backward: 4 (one CTA per SM; the dgamma partials share the
// registers).  Forward: 4 (two CTAs per SM) while that takes at most 16
// CTAs, else 16 (8 with a residual or float32 weights).  Measured on GB300
// (bf16, 256 MiB of rows): the backward with 4 vectors ran at 86 % of HBM at
// N = 32768 and 84 % at 65536 against 81 % and 78 % with 2 (twice the
// slices, two CTAs per SM); the forward at N = 131072 at 85 % with 8 slices
// of 4 against 62 % with 2 of 16.
static int64_t slices(int64_t NV, int kv) {
  return (NV + (int64_t)kv * rmsk::kWideThreads - 1) / ((int64_t)kv * rmsk::kWideThreads);
}
static int wide_kv(int64_t NV, int dtype, bool bwd, bool res) {
  const int gv_bytes = (dtype == kBF16W32 || dtype == kF16W32) ? 32 : 16;
  if (slices(NV, 4) <= rmsk::kWideMaxCluster) return 4;
  if (bwd) return 0;
  const int kv = (res || gv_bytes == 32) ? 8 : 16;
  if (slices(NV, kv) <= rmsk::kWideMaxCluster &&
      (int64_t)kv * rmsk::kWideThreads * gv_bytes <= rmsk::kWideGammaSmem)
    return kv;
  return 0;
}

bool plan_chunked(int N, int dtype, bool bwd, bool res, Mapping* m) {
  const int64_t row_bytes = (int64_t)N * dtype_bytes(dtype);
  if (N <= 0 || row_bytes % 16 != 0) return false;
  const int64_t NV = row_bytes / 16;
  m->path = kChunked;
  m->rows_per_cta = 1;
  const int kv = wide_kv(NV, dtype, bwd, res);
  if (kv > 0) {
    const int gv_bytes = (dtype == kBF16W32 || dtype == kF16W32) ? 32 : 16;
    m->wide = 1;
    m->kv = kv;
    m->threads = rmsk::kWideThreads;
    m->G = rmsk::kWideThreads;
    m->sv = kv * rmsk::kWideThreads;
    m->cluster = (int)((NV + m->sv - 1) / m->sv);
    m->chunks = 0;
    m->smem = (size_t)m->sv * gv_bytes;
    return true;
  }
  m->wide = 0;
  m->cluster = 1;
  m->threads = rmsk::kChunkThreads;
  m->kv = rmsk::kChunkVecs;
  m->G = rmsk::kChunkThreads;
  m->chunks = (int)((NV + rmsk::kChunkSpan - 1) / rmsk::kChunkSpan);
  m->smem = 0;
  return true;
}

// Launch configuration of the one-pass kernels: programmatic serialisation
// and, for C > 1, the cluster dimension.
struct WideLaunch {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  WideLaunch(const Mapping& m, int64_t grid, cudaStream_t s) {
    cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(m.threads);
    cfg.dynamicSmemBytes = m.smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
    if (m.cluster > 1) {
      attr[1].id = cudaLaunchAttributeClusterDimension;
      attr[1].val.clusterDim.x = m.cluster;
      attr[1].val.clusterDim.y = 1;
      attr[1].val.clusterDim.z = 1;
      cfg.numAttrs = 2;
    }
    cfg.attrs = attr;
  }
};

namespace {
struct ClusterFit {
  const void* k;
  int dev, C;
  size_t smem;
  int n;
};
std::mutex g_fit_mu;
ClusterFit g_fit[64];
int g_fit_n = 0;
}  // namespace

// How many clusters of m.cluster CTAs of kernel k are resident at once
// (cached per kernel, device, cluster size and shared memory).  The kernel
// is opted in to the device's full shared memory and, above 8 CTAs, to
// non-portable cluster sizes, once.
static cudaError_t wide_units(const void* k, const Mapping& m, const DeviceInfo& d, int* units) {
  std::lock_guard<std::mutex> lk(g_fit_mu);
  for (int i = 0; i < g_fit_n; ++i) {
    const ClusterFit& f = g_fit[i];
    if (f.k == k && f.dev == d.device && f.C == m.cluster && f.smem == m.smem) {
      *units = f.n;
      return cudaSuccess;
    }
  }
  cudaError_t e = opt_in_max_smem(k, d);
  if (e != cudaSuccess) return e;
  if (m.cluster > 8) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  int n = 0;
  if (m.cluster > 1) {
    WideLaunch L(m, m.cluster, nullptr);
    e = cudaOccupancyMaxActiveClusters(&n, k, &L.cfg);
  } else {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, m.threads, m.smem);
    n *= d.sms;
  }
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  if (g_fit_n < 64) g_fit[g_fit_n++] = ClusterFit{k, d.device, m.cluster, m.smem, n};
  *units = n;
  return cudaSuccess;
}

template <typename T, typename W, bool GEMMA, bool RES>
static const void* wide_fwd_kernel(int kv) {
  switch (kv) {
    case 4: return reinterpret_cast<const void*>(&rmsk::rms_fwd_wide_kernel<T, W, 4, GEMMA, RES>);
    case 8: return reinterpret_cast<const void*>(&rmsk::rms_fwd_wide_kernel<T, W, 8, GEMMA, RES>);
    case 16:
      if constexpr (!RES && sizeof(rmsk::GammaVec<T, W>) == 16)
        return reinterpret_cast<const void*>(&rmsk::rms_fwd_wide_kernel<T, W, 16, GEMMA, RES>);
      return nullptr;
  }
  return nullptr;
}

template <typename T, typename W, bool GEMMA, bool RES>
static const void* wide_bwd_kernel() {
  return reinterpret_cast<const void*>(&rmsk::rms_bwd_wide_kernel<T, W, GEMMA, RES>);
}

static rmsk::WideParams wide_params(const Mapping& m, int64_t M, int N) {
  rmsk::WideParams p{};
  p.M = M;
  p.N = N;
  p.C = m.cluster;
  p.SV = m.sv;
  return p;
}

static cudaError_t launch_fwd_wide(const FwdArgs& a, const Mapping& m, const DeviceInfo& d,
                                   long long wait_limit, cudaStream_t s) {
  return rmsk::with_types(a.dtype, a.gemma, a.res != nullptr,
                         [&](auto* tp, auto* wp, auto gm, auto rs) -> cudaError_t {
    using T = std::remove_pointer_t<decltype(tp)>;
    using W = std::remove_pointer_t<decltype(wp)>;
    constexpr bool GEMMA = decltype(gm)::value;
    constexpr bool RES = decltype(rs)::value;
    const void* k = wide_fwd_kernel<T, W, GEMMA, RES>(m.kv);
    if (!k) return cudaErrorInvalidValue;
    int units = 0;
    cudaError_t e = wide_units(k, m, d, &units);
    if (e != cudaSuccess) return e;
    const int64_t U = std::min<int64_t>(units, a.M);
    rmsk::WideParams p = wide_params(m, a.M, a.N);
    p.x = a.x;
    p.gamma = a.gamma;
    p.in2 = a.res;
    p.out = a.y;
    p.h = a.h;
    p.rstd = a.rstd;
    p.eps = a.eps;
    p.wait_limit = wait_limit;
    WideLaunch L(m, U * m.cluster, s);
    void* args[] = {&p};
    return cudaLaunchKernelExC(&L.cfg, k, args);
  });
}

// The E4M3 cluster forward: slices of four vectors per thread in CTAs of
// RMS_QUANT_WIDE_THREADS threads (512 when a row needs more than 16 such
// slices), up to 16 slices a row; each CTA holds its weights and the row's
// slice in shared memory.  Its row chain (two exchanges and three passes)
// is long, so smaller CTAs, more of them on an SM, keep more rows in flight.
#ifndef RMS_QUANT_WIDE_THREADS
#define RMS_QUANT_WIDE_THREADS 256
#endif
bool plan_quant_wide(int N, int dtype, Mapping* m) {
  const int64_t row_bytes = (int64_t)N * dtype_bytes(dtype);
  if (N <= 0 || row_bytes % 16 != 0) return false;
  const int64_t NV = row_bytes / 16;
  int TPB = RMS_QUANT_WIDE_THREADS;
  int64_t C = (NV + 4 * TPB - 1) / (4 * TPB);
  if (C > rmsk::kWideMaxCluster) {
    TPB = 512;
    C = (NV + 4 * TPB - 1) / (4 * TPB);
  }
  if (C > rmsk::kWideMaxCluster) return false;  // a CTA per row
  const int64_t sv = 4 * (int64_t)TPB;
  const int gv_bytes = (dtype == kBF16W32 || dtype == kF16W32) ? 32 : 16;
  m->path = kChunked;
  m->rows_per_cta = 1;
  m->wide = 1;
  m->kv = 4;
  m->threads = TPB;
  m->G = TPB;
  m->sv = (int)sv;
  m->cluster = (int)C;
  m->chunks = 0;
  m->smem = (size_t)sv * (gv_bytes + 16);  // the weights and the row's slice
  return true;
}

cudaError_t launch_fwd_quant_wide(const QuantArgs& a, const Mapping& m, const DeviceInfo& d,
                                  long long wait_limit, cudaStream_t s) {
  return rmsk::with_types(a.dtype, a.gemma, false,
                         [&](auto* tp, auto* wp, auto gm, auto) -> cudaError_t {
    using T = std::remove_pointer_t<decltype(tp)>;
    using W = std::remove_pointer_t<decltype(wp)>;
    constexpr bool GEMMA = decltype(gm)::value;
    const void* k =
        m.threads == 512
            ? reinterpret_cast<const void*>(&rmsk::rms_fwd_quant_wide_kernel<T, W, GEMMA, 512>)
            : reinterpret_cast<const void*>(
                  &rmsk::rms_fwd_quant_wide_kernel<T, W, GEMMA, RMS_QUANT_WIDE_THREADS>);
    int units = 0;
    cudaError_t e = wide_units(k, m, d, &units);
    if (e != cudaSuccess) return e;
    const int64_t U = std::min<int64_t>(units, a.M);
    rmsk::WideParams p = wide_params(m, a.M, a.N);
    p.x = a.x;
    p.gamma = a.gamma;
    p.out = a.q;
    p.h = a.scale;
    p.rstd = a.rstd;
    p.eps = a.eps;
    p.wait_limit = wait_limit;
    WideLaunch L(m, U * m.cluster, s);
    void* args[] = {&p};
    return cudaLaunchKernelExC(&L.cfg, k, args);
  });
}

// The three-pass row pass: C CTAs per row (a cluster), C doubling from 1
// while the rows alone give fewer than 4 CTAs per SM and each CTA keeps at
// least two chunks of the row; one row per cluster at a time, grid-strided.
namespace {
std::mutex g_c16_mu;
const void* g_c16[64];
int g_c16_n = 0;
}  // namespace

static cudaError_t allow_cluster16(const void* k) {
  std::lock_guard<std::mutex> lk(g_c16_mu);
  for (int i = 0; i < g_c16_n; ++i)
    if (g_c16[i] == k) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess && g_c16_n < 64) g_c16[g_c16_n++] = k;
  return e;
}

template <typename T, typename W, bool GEMMA, bool BWD, bool RES>
static cudaError_t launch_rowstat(const T* x, const T* dy, const W* g, const float* rstd_in,
                                  float* out, int64_t M, int N, float eps, const T* res, T* h,
                                  const DeviceInfo& d, cudaStream_t s) {
  const int64_t NV = (int64_t)N * sizeof(T) / 16;
  int C = 1;
  while (C < rmsk::kWideMaxCluster && M * C < 4ll * d.sms &&
         (int64_t)(2 * C) * 2 * rmsk::kChunkSpan <= NV)
    C *= 2;
  const int SV = (int)((NV + C - 1) / C);
  auto* k = rmsk::rms_rowstat_kernel<T, W, GEMMA, BWD, RES>;
  if (C == 1) {
    const int64_t grid = std::min<int64_t>(M, (int64_t)d.sms * 4);
    return rmsk::launch_pdl(k, dim3((unsigned)grid), dim3(rmsk::kChunkThreads), 0, s, x, dy, g,
                            rstd_in, out, M, N, eps, res, h, 1, SV);
  }
  if (C > 8) {
    const cudaError_t e = allow_cluster16(reinterpret_cast<const void*>(k));
    if (e != cudaSuccess) return e;
  }
  const int64_t clusters = std::min<int64_t>(M, 65536);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * C));
  cfg.blockDim = dim3(rmsk::kChunkThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, x, dy, g, rstd_in, out, M, N, eps, res, h, C, SV);
}

cudaError_t launch_fwd_chunked(const FwdArgs& a, const Mapping& m, const DeviceInfo& d,
                               long long wait_limit, cudaStream_t s) {
  if (m.wide) return launch_fwd_wide(a, m, d, wait_limit, s);
  return rmsk::with_types(a.dtype, a.gemma, a.res != nullptr,
                         [&](auto* tp, auto* wp, auto gm, auto rs) -> cudaError_t {
    using T = std::remove_pointer_t<decltype(tp)>;
    using W = std::remove_pointer_t<decltype(wp)>;
    constexpr bool GEMMA = decltype(gm)::value;
    constexpr bool RES = decltype(rs)::value;
    const T* x = static_cast<const T*>(a.x);
    const W* g = static_cast<const W*>(a.gamma);
    cudaError_t e = launch_rowstat<T, W, GEMMA, false, RES>(
        x, (const T*)nullptr, g, (const float*)nullptr, a.rstd, a.M, a.N, a.eps,
        static_cast<const T*>(a.res), static_cast<T*>(a.h), d, s);
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
// The one-pass backward kernel of a call.
static const void* wide_bwd_for(const BwdArgs& a) {
  const void* k = nullptr;
  rmsk::with_types(a.dtype, a.gemma, a.dh != nullptr,
                   [&](auto* tp, auto* wp, auto gm, auto rs) -> cudaError_t {
    using T = std::remove_pointer_t<decltype(tp)>;
    using W = std::remove_pointer_t<decltype(wp)>;
    k = wide_bwd_kernel<T, W, decltype(gm)::value, decltype(rs)::value>();
    return cudaSuccess;
  });
  return k;
}

bool size_bwd_chunked(const BwdArgs& a, const DeviceInfo& d, Mapping* m, float** kbuf) {
  const int64_t cap = std::min<int64_t>(a.M, max_partials(d.sms));  // workspace rows
  if (m->wide) {  // one workspace row per cluster; no per-row values to keep
    int units = 0;
    if (wide_units(wide_bwd_for(a), *m, d, &units) != cudaSuccess) return false;
    const int64_t U = std::max<int64_t>(1, std::min<int64_t>(units, cap));
    m->partials = U;
    m->blocks = U * m->cluster;
    *kbuf = nullptr;
    return true;
  }
  int64_t RG = std::max<int64_t>(1, max_partials(d.sms) / m->chunks);
  if (a.M <= a.N) {
    *kbuf = a.dgamma;
  } else {
    const int64_t krows = (a.M + a.N - 1) / a.N;
    if (cap - krows < 1) return false;  // many short rows: not this mapping's shape
    RG = std::min<int64_t>(RG, cap - krows);
    *kbuf = a.ws ? a.ws + (cap - krows) * (int64_t)a.N : nullptr;
  }
  RG = std::max<int64_t>(1, std::min<int64_t>(RG, cap));
  if (RG * m->chunks > INT32_MAX) return false;
  m->partials = RG;
  m->blocks = RG * m->chunks;
  return true;
}

cudaError_t launch_bwd_chunked(const BwdArgs& a, const Mapping& m, float* kbuf,
                               const DeviceInfo& d, long long wait_limit, cudaStream_t s) {
  if (m.wide) {
    rmsk::WideParams p = wide_params(m, a.M, a.N);
    p.x = a.x;
    p.gamma = a.gamma;
    p.in2 = a.dy;
    p.in3 = a.dh;
    p.out = a.dx;
    p.rstd = const_cast<float*>(a.rstd);
    p.ws = a.ws;
    p.wait_limit = wait_limit;
    WideLaunch L(m, m.blocks, s);
    void* args[] = {&p};
    return cudaLaunchKernelExC(&L.cfg, wide_bwd_for(a), args);
  }
  return rmsk::with_types(a.dtype, a.gemma, a.dh != nullptr,
                         [&](auto* tp, auto* wp, auto gm, auto rs) -> cudaError_t {
    using T = std::remove_pointer_t<decltype(tp)>;
    using W = std::remove_pointer_t<decltype(wp)>;
    constexpr bool GEMMA = decltype(gm)::value;
    constexpr bool RES = decltype(rs)::value;
    const T* x = static_cast<const T*>(a.x);
    const T* dy = static_cast<const T*>(a.dy);
    const W* g = static_cast<const W*>(a.gamma);
    cudaError_t e = launch_rowstat<T, W, GEMMA, true, false>(
        x, dy, g, a.rstd, kbuf, a.M, a.N, 0.f, (const T*)nullptr, (T*)nullptr, d, s);
    if (e != cudaSuccess) return e;
    return rmsk::launch_pdl(rmsk::rms_bwd_chunk_kernel<T, W, GEMMA, RES>, dim3((unsigned)m.blocks),
                      dim3(rmsk::kChunkThreads), 0, s, dy, x, g, a.rstd, (const float*)kbuf,
                      static_cast<T*>(a.dx), a.ws, a.M, a.N, m.chunks, m.partials,
                      static_cast<const T*>(a.dh));
  });
}

cudaError_t take_wide_device_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, rmsk::g_wide_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(rmsk::g_wide_device_status, &zero, sizeof(int));
    if (e != cudaSuccess) return e;
  }
  *status = v;
  return cudaSuccess;
}

}  // namespace rmsi
