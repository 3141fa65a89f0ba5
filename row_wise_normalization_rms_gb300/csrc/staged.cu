// Staged mapping: persistent CTAs stream tiles of R consecutive rows
// (R * N contiguous elements) from HBM into an S-deep ring of shared-memory
// stages with bulk TMA copies (cp.async.bulk + mbarrier), so S-1 tiles are
// always in flight no matter how long the math on the current tile takes.
// A group of G threads owns one row of the tile; each thread moves its
// 16-byte vectors from the stage into registers, the group reduces, and the
// results go straight to global memory.  The stage is handed back to the
// copy engine as soon as every thread has read it (one barrier per tile,
// which the row reduction needs anyway).
//
// Forward computes r and y exactly as the register mapping does; backward
// stages x and dy together and accumulates dgamma column partials in
// registers across the CTA's tiles (static tile order), one workspace row
// per CTA.
//
// Every mbarrier wait is bounded.  If a wait gives up, the CTA stops
// consuming tiles, waits (again bounded) for the copies it has in flight,
// sets the device status word and exits; the host reads that word through
// rms_last_device_status().  Nothing spins without a limit.
//
// Sources: "Hướng dẫn Triton RMSNorm: kernel, backward…" (formulas, true-N
// mean, per-part dgamma partials reduced in a second pass); "第 07 章:
// LayerNorm——反向传播与原子锁", step 3 (a row too wide for one block is
// walked through in chunks; here it is staged whole in shared memory).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace rmsk {

// Nonzero once a bounded wait gave up; read and cleared by the host.
__device__ int g_rms_device_status = 0;

constexpr int kHeaderBytes = 1024;  // barriers, reduction slots, abort flags

// Kernel arguments, kept within 128 bytes: at 152 bytes (three more
// pointers) the backward measured 2-7 % slower on GB300 at several shapes
// with no other change, so the roles of the two directions share fields.
struct StagedParams {
  const void* x;
  const void* gamma;
  const void* in2;  // backward: dy; fused forward: the residual (staged beside x)
  const void* in3;  // fused backward: dh (staged after dy)
  void* out;        // forward: y; backward: dx (may equal dy, or dh)
  void* h;          // fused forward: h = x + residual (may equal the residual)
  float* rstd;      // forward: written; backward: read
  float* ws;        // backward: [units][N] column partials
  int64_t M;
  int N;
  float eps;
  int G;   // threads per row slice
  int R;   // rows per tile (1 when C > 1)
  int S;   // stages
  int C;   // CTAs per cluster sharing one row (1: no cluster)
  int SV;  // 16-byte vectors per CTA's column slice (the whole row when C == 1)
  uint32_t tile_bytes;   // R * SV * 16
  uint32_t stage_bytes;  // tile_bytes times the tensors staged (x; dy; residual or dh)
  long long wait_limit;
  int64_t ntiles;
};
static_assert(sizeof(StagedParams) <= 128, "staged kernel arguments grew past 128 bytes");

struct StageHeader {
  uint64_t* full;
  float* red;             // [2][32] warp partial sums
  volatile int* abort;    // [2] a wait of this CTA gave up
  float* sum_in;          // [2][16] row partials pushed by the cluster's CTAs, by rank
  int* abort_in;          // [2][16] their abort flags
  uint8_t* stages;
};

__device__ __forceinline__ StageHeader header(uint8_t* smem) {
  StageHeader h;
  h.full = reinterpret_cast<uint64_t*>(smem);
  h.red = reinterpret_cast<float*>(smem + 64);
  h.abort = reinterpret_cast<volatile int*>(smem + 320);
  h.sum_in = reinterpret_cast<float*>(smem + 384);
  h.abort_in = reinterpret_cast<int*>(smem + 512);
  h.stages = smem + kHeaderBytes;
  return h;
}

// Which part of which rows this CTA works on.  Without clusters a unit is a
// CTA and its slice is the whole row; with clusters of C CTAs a unit is a
// cluster and CTA rank c owns vectors [c*SV, c*SV + nvs) of each row.
struct Slice {
  int64_t unit, units;  // this work unit and how many there are
  int rank;             // CTA rank in the cluster (0 without clusters)
  int v0, nvs;          // first vector and vector count of this CTA's slice
};

__device__ __forceinline__ Slice my_slice(const StagedParams& p, int NV) {
  Slice sl;
  sl.rank = p.C > 1 ? (int)cluster_rank() : 0;
  sl.unit = blockIdx.x / p.C;
  sl.units = gridDim.x / p.C;
  sl.v0 = sl.rank * p.SV;
  sl.nvs = min(p.SV, NV - sl.v0);
  return sl;
}

// Thread 0: start the copy of local tile i (rows of tile unit + i*units,
// this CTA's slice) into stage i % S: NT tensors one after the other, x
// first, then t1 (dy for the backward, the residual for a fused forward)
// and t2 (dh for a fused backward).
template <typename T, int NT, bool BWD>
__device__ __forceinline__ void issue_tile(const StagedParams& p, const StageHeader& h,
                                           const Slice& sl, int64_t i, uint64_t pol) {
  const int64_t t = sl.unit + i * sl.units;
  const int64_t row0 = t * p.R;
  const int64_t rows = min((int64_t)p.R, p.M - row0);
  const int64_t row_bytes = (int64_t)p.N * sizeof(T);
  // Without clusters nvs*16 == row_bytes and the R rows are contiguous.
  const uint32_t bytes = (uint32_t)(rows * sl.nvs * 16);
  const int64_t src = row0 * row_bytes + (int64_t)sl.v0 * 16;
  const int s = (int)(i % p.S);
  const uint32_t bar = smem_u32(&h.full[s]);
  const uint32_t dst = smem_u32(h.stages + (size_t)s * p.stage_bytes);
  mbar_arrive_expect_tx(bar, NT * bytes);
  tma_load_1d(dst, static_cast<const char*>(p.x) + src, bytes, bar, pol);
  if (NT > 1)
    tma_load_1d(dst + p.tile_bytes, static_cast<const char*>(p.in2) + src, bytes, bar,
                pol);
  if (NT > 2)
    tma_load_1d(dst + 2 * p.tile_bytes, static_cast<const char*>(p.in3) + src, bytes, bar, pol);
}

// After an abort at local tile i: wait (bounded) for the copies this CTA
// issued and has not consumed (tiles i .. issued-1), then raise the device
// status.  Thread 0 only.
__device__ __forceinline__ void drain_and_flag(const StagedParams& p, const StageHeader& h,
                                               int64_t i, int64_t issued) {
  for (int64_t j = i; j < issued; ++j)
    mbar_wait(smem_u32(&h.full[j % p.S]), (uint32_t)((j / p.S) & 1), kDrainPolls);
  g_rms_device_status = 1;
  __threadfence();
}

__device__ __forceinline__ void init_barriers(const StagedParams& p, const StageHeader& h) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.S; ++s) mbar_init(smem_u32(&h.full[s]), 1);
    h.abort[0] = 0;
    h.abort[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();
}

// The row's total of a per-thread partial, after the stage barrier of
// iteration i.  Without clusters: the group's warp partials in warp order.
// With clusters (one row per tile, the CTA is one group): thread c pushes
// this CTA's sum and abort flag into slot [buf][rank] of CTA c, one cluster
// barrier later every CTA adds the C slots in rank order from its own shared
// memory (the same total everywhere) and makes the same abort decision, so
// all CTAs of a cluster leave the loop together.  A slot [buf] is written
// again two tiles later, after the next barrier, which no CTA passes before
// every CTA has read it.  Returns the total; *abort tells whether any CTA
// (of the cluster) gave up a wait.
__device__ __forceinline__ float row_total(const StagedParams& p, const StageHeader& h, int buf,
                                           int first_warp, int nw, int rank, bool* abort) {
  float tot = 0.f;
  for (int w = 0; w < nw; ++w) tot += h.red[buf * 32 + first_warp + w];
  if (p.C == 1) {
    *abort = h.abort[buf] != 0;
    return tot;
  }
  if ((int)threadIdx.x < p.C) {
    const uint32_t c = threadIdx.x;
    st_cluster_f32(map_to_rank(smem_u32(&h.sum_in[buf * 16 + rank]), c), tot);
    st_cluster_s32(map_to_rank(smem_u32(&h.abort_in[buf * 16 + rank]), c), h.abort[buf]);
  }
  cluster_sync();
  float all = 0.f;
  int ab = 0;
  for (int c = 0; c < p.C; ++c) {
    all += h.sum_in[buf * 16 + c];
    ab |= h.abort_in[buf * 16 + c];
  }
  *abort = ab != 0;
  return all;
}

// Pipeline shared by both kernels.  Local tile i lives in stage i % S.
// Iteration i: wait for tile i, first pass over it (row partial sums),
// barrier, second pass (outputs).  The barrier of iteration i also proves
// every thread of the CTA finished the second pass of tile i-1, so right
// after it thread 0 refills that stage with the next tile: S-2 tiles stay in
// flight while tile i is processed, and no row slice has to stay in
// registers across the barrier.  With clusters a cluster barrier follows for
// the exchange of row partials, and a last one before exit keeps every CTA's
// shared memory alive while its peers may still read it.

// With RES the residual is staged beside x; the first pass forms h = x +
// res, stores it and reduces it, the second forms it again from the stage
// (at most 512 threads: twice the vectors per thread are live).
template <typename T, typename W, int KV, bool GEMMA, bool RES>
__global__ void __launch_bounds__(RES ? 512 : 1024)
rms_fwd_staged_kernel(const StagedParams p) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  extern __shared__ __align__(128) uint8_t smem[];
  const StageHeader h = header(smem);
  const int NV = p.N / VN;
  const Slice sl = my_slice(p, NV);
  const int q = threadIdx.x / p.G;
  const int lig = threadIdx.x - q * p.G;
  const int warp = threadIdx.x >> 5;
  const int first_warp = q * (p.G >> 5);
  const int nw = p.G >> 5;
  const int64_t my_tiles = (p.ntiles - sl.unit + sl.units - 1) / sl.units;
  const uint32_t row_off = (uint32_t)(q * p.SV * 16);

  init_barriers(p, h);
  pdl_wait();
  uint64_t pol = 0;
  int64_t issued = 0;  // thread 0 only
  if (threadIdx.x == 0) {
    pol = l2_evict_first_policy();
    const int64_t pre = min((int64_t)p.S, my_tiles);
    for (; issued < pre; ++issued) issue_tile<T, RES ? 2 : 1, false>(p, h, sl, issued, pol);
  }

  GV gw[KV];
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = lig + k * p.G;
    gw[k] = v < sl.nvs ? GV::load(p.gamma, sl.v0 + v) : GV::zero();
  }

  int64_t i = 0;
  bool aborted = false;
  int s = 0;               // i % S, kept as a counter (no 64-bit division per tile)
  uint32_t parity = 0;     // (i / S) & 1
  for (; i < my_tiles; ++i, s = (s + 1 == p.S) ? 0 : s + 1, parity ^= (s == 0)) {
    const int buf = (int)(i & 1);
    const int64_t row = (sl.unit + i * sl.units) * p.R + q;
    const bool active = row < p.M;
    if (!mbar_wait(smem_u32(&h.full[s]), parity, p.wait_limit)) h.abort[buf] = 1;

    const uint32_t xs = smem_u32(h.stages + (size_t)s * p.stage_bytes) + row_off;
    f32x2 ss2 = 0ull;
    if (active) {
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int v = lig + k * p.G;
        if (v < sl.nvs) {
          if (RES) {
            const uint4 hv = Math::add_round(lds128(xs + 16u * v),
                                             lds128(xs + p.tile_bytes + 16u * v));
            st_stream(reinterpret_cast<uint4*>(p.h) + row * (int64_t)NV + sl.v0 + v, hv);
            Math::sumsq(hv, ss2);
          } else {
            Math::sumsq(lds128(xs + 16u * v), ss2);
          }
        }
      }
    }
    const float ss = warp_sum(lo2(ss2) + hi2(ss2));
    if ((threadIdx.x & 31) == 0) h.red[buf * 32 + warp] = ss;
    __syncthreads();  // partial sums visible; tile i-1 fully consumed
    if (threadIdx.x == 0 && i >= 1 && issued < my_tiles && !h.abort[buf])
      issue_tile<T, RES ? 2 : 1, false>(p, h, sl, issued++, pol);
    bool abort;
    const float tot = row_total(p, h, buf, first_warp, nw, sl.rank, &abort);
    if (abort) {
      aborted = true;
      break;
    }
    const float r = 1.0f / sqrtf(tot / (float)p.N + p.eps);
    if (active) {
      if (lig == 0 && sl.rank == 0) p.rstd[row] = r;
      uint4* yr = reinterpret_cast<uint4*>(p.out) + row * (int64_t)NV + sl.v0;
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int v = lig + k * p.G;
        if (v < sl.nvs) {
          if (RES) {
            st_stream(yr + v, Math::forward(Math::add_round(lds128(xs + 16u * v),
                                                            lds128(xs + p.tile_bytes + 16u * v)),
                                            gw[k], r));
          } else {
            st_stream(yr + v, Math::forward(lds128(xs + 16u * v), gw[k], r));
          }
        }
      }
    }
  }
  if (aborted && threadIdx.x == 0) drain_and_flag(p, h, i, issued);
  if (p.C > 1) cluster_sync();
}

// With RES, dh is staged after dy and added to dx before its rounding.
template <typename T, typename W, int KV, bool GEMMA, bool RES>
__global__ void __launch_bounds__(512)
rms_bwd_staged_kernel(const StagedParams p) {
  using Math = RowMath<T, W, GEMMA>;
  using GV = GammaVec<T, W>;
  constexpr int VN = Elem<T>::kPerVec;
  constexpr int NP = Math::kPairs;
  extern __shared__ __align__(128) uint8_t smem[];
  const StageHeader h = header(smem);
  const int NV = p.N / VN;
  const Slice sl = my_slice(p, NV);
  const int q = threadIdx.x / p.G;
  const int lig = threadIdx.x - q * p.G;
  const int warp = threadIdx.x >> 5;
  const int first_warp = q * (p.G >> 5);
  const int nw = p.G >> 5;
  const int64_t my_tiles = (p.ntiles - sl.unit + sl.units - 1) / sl.units;
  const uint32_t row_off = (uint32_t)(q * p.SV * 16);

  init_barriers(p, h);
  pdl_wait();
  uint64_t pol = 0;
  int64_t issued = 0;  // thread 0 only
  if (threadIdx.x == 0) {
    pol = l2_evict_first_policy();
    const int64_t pre = min((int64_t)p.S, my_tiles);
    for (; issued < pre; ++issued) issue_tile<T, RES ? 3 : 2, true>(p, h, sl, issued, pol);
  }

  GV gw[KV];
  f32x2 acc[KV][NP];
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int v = lig + k * p.G;
    gw[k] = v < sl.nvs ? GV::load(p.gamma, sl.v0 + v) : GV::zero();
#pragma unroll
    for (int e = 0; e < NP; ++e) acc[k][e] = 0ull;
  }

  int64_t i = 0;
  bool aborted = false;
  int s = 0;               // i % S, kept as a counter (no 64-bit division per tile)
  uint32_t parity = 0;     // (i / S) & 1
  for (; i < my_tiles; ++i, s = (s + 1 == p.S) ? 0 : s + 1, parity ^= (s == 0)) {
    const int buf = (int)(i & 1);
    const int64_t row = (sl.unit + i * sl.units) * p.R + q;
    const bool active = row < p.M;
    const float r = active ? p.rstd[row] : 0.f;
    if (!mbar_wait(smem_u32(&h.full[s]), parity, p.wait_limit)) h.abort[buf] = 1;

    const uint32_t xs = smem_u32(h.stages + (size_t)s * p.stage_bytes) + row_off;
    const uint32_t ds = xs + p.tile_bytes;
    // First pass: r*sum(u*x) over the slice, and the slice's dgamma terms.
    f32x2 sux2 = 0ull;
    if (active) {
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int v = lig + k * p.G;
        if (v < sl.nvs)
          Math::backward_sums(lds128(xs + 16u * v), lds128(ds + 16u * v), gw[k], r, sux2, acc[k]);
      }
    }
    const float sux = warp_sum(lo2(sux2) + hi2(sux2));
    if ((threadIdx.x & 31) == 0) h.red[buf * 32 + warp] = sux;
    __syncthreads();  // partial sums visible; tile i-1 fully consumed
    if (threadIdx.x == 0 && i >= 1 && issued < my_tiles && !h.abort[buf])
      issue_tile<T, RES ? 3 : 2, true>(p, h, sl, issued++, pol);
    bool abort;
    const float tot = row_total(p, h, buf, first_warp, nw, sl.rank, &abort);
    if (abort) {
      aborted = true;
      break;
    }
    const float kc = tot / (float)p.N;  // r * mean(u*x)
    // Second pass: dx = r*(u - x*r*kc).
    if (active) {
      uint4* out = reinterpret_cast<uint4*>(p.out) + row * (int64_t)NV + sl.v0;
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int v = lig + k * p.G;
        if constexpr (RES) {
          if (v < sl.nvs)
            st_stream(out + v, Math::backward_dx_add(lds128(xs + 16u * v), lds128(ds + 16u * v),
                                                     gw[k], r, kc,
                                                     lds128(ds + p.tile_bytes + 16u * v)));
        } else {
          if (v < sl.nvs)
            st_stream(out + v, Math::backward_dx(lds128(xs + 16u * v), lds128(ds + 16u * v), gw[k], r, kc));
        }
      }
    }
  }
  if (aborted) {
    if (threadIdx.x == 0) drain_and_flag(p, h, i, issued);
    if (p.C > 1) cluster_sync();
    return;  // the partial row stays unwritten; the status word reports it
  }

  // This unit's column partials: one workspace row per unit; this CTA writes
  // its slice; groups of a CTA (several rows per tile) are combined in group
  // order through the (now idle) stage memory.
  float* wp = p.ws + sl.unit * (int64_t)p.N + (int64_t)sl.v0 * VN;
  if (p.R == 1) {
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = lig + k * p.G;
      if (v < sl.nvs) {
        float4* w4 = reinterpret_cast<float4*>(wp + (int64_t)v * VN);
#pragma unroll
        for (int c = 0; c < NP / 2; ++c)
          w4[c] = make_float4(lo2(acc[k][2 * c]), hi2(acc[k][2 * c]), lo2(acc[k][2 * c + 1]),
                              hi2(acc[k][2 * c + 1]));
      }
    }
  } else {
    float* part = reinterpret_cast<float*>(h.stages);  // [R][N] fits in the stage ring
    __syncthreads();
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int v = lig + k * p.G;
      if (v < sl.nvs) {
#pragma unroll
        for (int e = 0; e < NP; ++e) {
          part[(int64_t)q * p.N + v * VN + 2 * e] = lo2(acc[k][e]);
          part[(int64_t)q * p.N + v * VN + 2 * e + 1] = hi2(acc[k][e]);
        }
      }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < p.N; j += blockDim.x) {
      float t = 0.f;
      for (int qq = 0; qq < p.R; ++qq) t += part[(int64_t)qq * p.N + j];
      wp[j] = t;
    }
  }
  if (p.C > 1) cluster_sync();
}

template <typename T, typename W, bool BWD, bool GEMMA, bool RES>
static const void* staged_ptr_g(int kv) {
  if (BWD) {
    switch (kv) {
      case 1: return reinterpret_cast<const void*>(&rms_bwd_staged_kernel<T, W, 1, GEMMA, RES>);
      case 2: return reinterpret_cast<const void*>(&rms_bwd_staged_kernel<T, W, 2, GEMMA, RES>);
      case 3: return reinterpret_cast<const void*>(&rms_bwd_staged_kernel<T, W, 3, GEMMA, RES>);
      case 4: return reinterpret_cast<const void*>(&rms_bwd_staged_kernel<T, W, 4, GEMMA, RES>);
    }
  } else {
    switch (kv) {
      case 1: return reinterpret_cast<const void*>(&rms_fwd_staged_kernel<T, W, 1, GEMMA, RES>);
      case 2: return reinterpret_cast<const void*>(&rms_fwd_staged_kernel<T, W, 2, GEMMA, RES>);
      case 4: return reinterpret_cast<const void*>(&rms_fwd_staged_kernel<T, W, 4, GEMMA, RES>);
    }
  }
  return nullptr;
}

template <typename T, typename W, bool BWD>
static const void* staged_ptr(int kv, bool gemma, bool res) {
  if (res) return gemma ? staged_ptr_g<T, W, BWD, true, true>(kv) : staged_ptr_g<T, W, BWD, false, true>(kv);
  return gemma ? staged_ptr_g<T, W, BWD, true, false>(kv) : staged_ptr_g<T, W, BWD, false, false>(kv);
}

}  // namespace rmsk

namespace rmsi {

namespace {

// Measured on GB300 over N = 512 .. 16384 bf16: up to four CTAs per SM
// sharing 224 KiB of stages is as fast or faster than fewer, larger rings.
#ifndef RMS_STAGED_SMEM_PER_SM
#define RMS_STAGED_SMEM_PER_SM (224 * 1024)
#endif
#ifndef RMS_STAGED_MAX_CTAS_PER_SM
#define RMS_STAGED_MAX_CTAS_PER_SM 4
#endif
#ifndef RMS_STAGED_TILE_BYTES
#define RMS_STAGED_TILE_BYTES 16384
#endif
#ifndef RMS_STAGED_MAX_STAGES
#define RMS_STAGED_MAX_STAGES 8
#endif
#ifndef RMS_STAGED_KV_MAX
#define RMS_STAGED_KV_MAX 4
#endif
#ifndef RMS_STAGED_MIN_CPS
#define RMS_STAGED_MIN_CPS 1
#endif
#ifndef RMS_STAGED_BWD_KV3
#define RMS_STAGED_BWD_KV3 1
#endif

const void* staged_kernel(int dtype, bool bwd, int kv, bool gemma, bool res) {
  switch (dtype) {
    case kBF16:
      return bwd ? rmsk::staged_ptr<__nv_bfloat16, __nv_bfloat16, true>(kv, gemma, res)
                 : rmsk::staged_ptr<__nv_bfloat16, __nv_bfloat16, false>(kv, gemma, res);
    case kF16:
      return bwd ? rmsk::staged_ptr<__half, __half, true>(kv, gemma, res)
                 : rmsk::staged_ptr<__half, __half, false>(kv, gemma, res);
    case kBF16W32:
      return bwd ? rmsk::staged_ptr<__nv_bfloat16, float, true>(kv, gemma, res)
                 : rmsk::staged_ptr<__nv_bfloat16, float, false>(kv, gemma, res);
    case kF16W32:
      return bwd ? rmsk::staged_ptr<__half, float, true>(kv, gemma, res)
                 : rmsk::staged_ptr<__half, float, false>(kv, gemma, res);
    default:
      return bwd ? rmsk::staged_ptr<float, float, true>(kv, gemma, res)
                 : rmsk::staged_ptr<float, float, false>(kv, gemma, res);
  }
}

// Occupancy per (kernel, device, threads, smem), so repeated calls make no
// driver queries.  Each kernel is opted in to the device's full dynamic
// shared memory once (the attribute is per kernel, last writer wins, so it
// is never lowered for a smaller configuration).
struct OccEntry {
  const void* k;
  int dev, threads;
  size_t smem;
  int occ;
};
std::mutex g_occ_mu;
OccEntry g_occ[128];
int g_occ_n = 0;

cudaError_t occupancy(const void* k, const DeviceInfo& d, int threads, size_t smem, int* occ) {
  std::lock_guard<std::mutex> lk(g_occ_mu);
  for (int i = 0; i < g_occ_n; ++i) {
    const OccEntry& e = g_occ[i];
    if (e.k == k && e.dev == d.device && e.threads == threads && e.smem == smem) {
      *occ = e.occ;
      return cudaSuccess;
    }
  }
  cudaError_t e = opt_in_max_smem(k, d);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, threads, smem);
  if (e != cudaSuccess) return e;
  if (g_occ_n < 128) g_occ[g_occ_n++] = OccEntry{k, d.device, threads, smem, *occ};
  return cudaSuccess;
}

}  // namespace

// One plan for a cluster size C: the row split into C slices of SV vectors
// (C = 1: whole rows, tiles of R rows of about 16 KiB, at most 16 rows), G
// threads per row slice with up to 4 vectors each, and as many stages as fit
// in the per-SM shared-memory budget, at least three per CTA (one being
// processed, one whose refill waits for the next barrier, one in flight):
// the most CTAs per SM, up to the cap, whose three stages fit.
static bool plan_for_cluster(int C, int NV, int64_t row_bytes, bool bwd, int tensors,
                             const DeviceInfo& d, Mapping* m, int64_t M) {
  if (C > 1 && NV < 64 * C) return false;  // rows this short never need a cluster
  const int SV = (NV + C - 1) / C;
  const int max_threads = (bwd || tensors > 1) ? 512 : 1024;
  int kv, G;
  if (SV <= 32) {
    kv = 1; G = 32;
  } else if (SV <= 64) {
    kv = 2; G = 32;
  } else {
    kv = RMS_STAGED_KV_MAX;
    G = ((SV + kv - 1) / kv + 31) / 32 * 32;
    if (G > max_threads) {
      kv = 4;
      G = ((SV + 3) / 4 + 31) / 32 * 32;
    }
    if (G > max_threads) return false;
  }
  // Rows per tile: a stage of about RMS_STAGED_TILE_BYTES per tensor of the
  // plain direction (x; x and dy) whatever the number of tensors staged (a
  // fused residual adds one), then halved while a persistent CTA would get
  // fewer than kMinTilesPerCta tiles (coarse tiles leave the last wave
  // ragged: Llama-7B-shaped 8192 x 4096 backward 38.9 -> 36.7 us on GB300).
  constexpr int64_t kMinTilesPerCta = 20;
  constexpr int64_t kMinTileBytes = 8192;  // per tensor: smaller tiles cost more than they save
  int R = 1;
  if (C == 1) {
    R = (int)((bwd ? 2 : 1) * RMS_STAGED_TILE_BYTES / tensors / row_bytes);
    if (R < 1) R = 1;
    if (R > 16) R = 16;
    while (R > 1 && G * R > max_threads) --R;
  }
  const int64_t budget = RMS_STAGED_SMEM_PER_SM;
  const int64_t cap = (int64_t)d.smem_optin - rmsk::kHeaderBytes;
  int64_t tile = 0, stage = 0;
  int cps = 0, S = 0;
  for (;;) {
    tile = (int64_t)R * SV * 16;
    stage = tensors * tile;
    cps = 0;
    for (int c = RMS_STAGED_MAX_CTAS_PER_SM; c >= 1; --c) {
      const int64_t per_cta = std::min(budget / c, cap);
      if (3 * stage <= per_cta) {
        cps = c;
        S = (int)(per_cta / stage);
        break;
      }
    }
    if (cps == 0 || R == 1 || M <= 0 || (R / 2) * row_bytes < kMinTileBytes) break;
    const int64_t tiles = (M + R - 1) / R;
    if (tiles >= kMinTilesPerCta * cps * d.sms) break;
    R /= 2;
  }
  if (cps == 0) return false;
  if (S > RMS_STAGED_MAX_STAGES) S = RMS_STAGED_MAX_STAGES;
  // A backward of whole rows at one CTA per SM has a row's warps to itself:
  // three vectors a thread instead of four give it a third more of them
  // where the row allows (10240 bf16: 448 threads instead of 320).
  if (RMS_STAGED_BWD_KV3 && bwd && C == 1 && R == 1 && cps == 1 && kv == 4) {
    const int G3 = ((SV + 2) / 3 + 31) / 32 * 32;
    if (G3 <= max_threads) {
      kv = 3;
      G = G3;
    }
  }
  m->path = kStaged;
  m->kv = kv;
  m->G = G;
  m->rows_per_cta = R;
  m->threads = G * R;
  m->stages = S;
  m->cluster = C;
  m->sv = SV;
  m->smem = rmsk::kHeaderBytes + (size_t)S * stage;
  m->blocks = cps;  // CTAs per SM wanted; the launcher turns it into a grid
  return true;
}

// The smallest cluster (1, 2, 4 or 8 CTAs) whose plan fits: rows up to
// 16 KiB (backward) or 64 KiB (forward) per CTA, so clusters take rows of
// up to 128 K bf16 elements in the backward and 256 K in the forward.
bool plan_staged(int N, int dtype, bool bwd, const DeviceInfo& d, Mapping* m, bool res,
                 int64_t M) {
  const int b = dtype_bytes(dtype);
  if (N <= 0 || ((int64_t)N * b) % 16 != 0) return false;
  const int64_t row_bytes = (int64_t)N * b;
  const int NV = (int)(row_bytes / 16);
  const int tensors = (bwd ? 2 : 1) + (res ? 1 : 0);  // x [, dy] [, residual or dh]
  for (int C = 1; C <= 8; C *= 2)
    if (plan_for_cluster(C, NV, row_bytes, bwd, tensors, d, m, M) && m->blocks >= RMS_STAGED_MIN_CPS)
      return true;
  for (int C = 1; C <= 8; C *= 2)
    if (plan_for_cluster(C, NV, row_bytes, bwd, tensors, d, m, M)) return true;
  return false;
}

// Launch config with programmatic serialisation and, for C > 1, the cluster
// dimension.
struct StagedLaunch {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  StagedLaunch(const Mapping& m, int64_t grid, cudaStream_t s) {
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

// Persistent grid: as many work units (CTAs, or clusters of C CTAs) as fit
// on the device at once, at most the planned CTAs per SM, at most the tiles.
static cudaError_t grid_for(const void* k, const Mapping& m, const DeviceInfo& d, int64_t ntiles,
                            int64_t* grid) {
  int occ = 0;
  cudaError_t e = occupancy(k, d, m.threads, m.smem, &occ);
  if (e != cudaSuccess) return e;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  int64_t units = std::min<int64_t>(occ, m.blocks) * d.sms / m.cluster;
  if (m.cluster > 1) {
    StagedLaunch L(m, m.cluster, nullptr);
    int nc = 0;
    e = cudaOccupancyMaxActiveClusters(&nc, k, &L.cfg);
    if (e != cudaSuccess) return e;
    if (nc < 1) return cudaErrorInvalidConfiguration;
    units = std::min<int64_t>(units, nc);
  }
  if (units > ntiles) units = ntiles;
  if (units < 1) units = 1;
  *grid = units * m.cluster;
  return cudaSuccess;
}

static rmsk::StagedParams params(const Mapping& m, int64_t M, int N, int tensors,
                                 long long wait_limit) {
  rmsk::StagedParams p{};
  p.M = M;
  p.N = N;
  p.G = m.G;
  p.R = m.rows_per_cta;
  p.S = m.stages;
  p.C = m.cluster;
  p.SV = m.sv;
  p.ntiles = (M + p.R - 1) / p.R;
  p.tile_bytes = (uint32_t)((int64_t)p.R * p.SV * 16);
  p.stage_bytes = tensors * p.tile_bytes;
  p.wait_limit = wait_limit;
  return p;
}

template <typename T, typename W, bool GEMMA, bool RES>
static cudaError_t launch_fwd_g(const rmsk::StagedParams& p, const Mapping& m, int64_t grid,
                                cudaStream_t s) {
  StagedLaunch L(m, grid, s);
  switch (m.kv) {
    case 1: return cudaLaunchKernelEx(&L.cfg, rmsk::rms_fwd_staged_kernel<T, W, 1, GEMMA, RES>, p);
    case 2: return cudaLaunchKernelEx(&L.cfg, rmsk::rms_fwd_staged_kernel<T, W, 2, GEMMA, RES>, p);
    case 4: return cudaLaunchKernelEx(&L.cfg, rmsk::rms_fwd_staged_kernel<T, W, 4, GEMMA, RES>, p);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, typename W, bool GEMMA, bool RES>
static cudaError_t launch_bwd_g(const rmsk::StagedParams& p, const Mapping& m, int64_t grid,
                                cudaStream_t s) {
  StagedLaunch L(m, grid, s);
  switch (m.kv) {
    case 1: return cudaLaunchKernelEx(&L.cfg, rmsk::rms_bwd_staged_kernel<T, W, 1, GEMMA, RES>, p);
    case 2: return cudaLaunchKernelEx(&L.cfg, rmsk::rms_bwd_staged_kernel<T, W, 2, GEMMA, RES>, p);
    case 3: return cudaLaunchKernelEx(&L.cfg, rmsk::rms_bwd_staged_kernel<T, W, 3, GEMMA, RES>, p);
    case 4: return cudaLaunchKernelEx(&L.cfg, rmsk::rms_bwd_staged_kernel<T, W, 4, GEMMA, RES>, p);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, typename W>
static cudaError_t launch_fwd_t(const rmsk::StagedParams& p, const Mapping& m, int64_t grid,
                                bool gemma, bool res, cudaStream_t s) {
  if (res)
    return gemma ? launch_fwd_g<T, W, true, true>(p, m, grid, s)
                 : launch_fwd_g<T, W, false, true>(p, m, grid, s);
  return gemma ? launch_fwd_g<T, W, true, false>(p, m, grid, s)
               : launch_fwd_g<T, W, false, false>(p, m, grid, s);
}

template <typename T, typename W>
static cudaError_t launch_bwd_t(const rmsk::StagedParams& p, const Mapping& m, int64_t grid,
                                bool gemma, bool res, cudaStream_t s) {
  if (res)
    return gemma ? launch_bwd_g<T, W, true, true>(p, m, grid, s)
                 : launch_bwd_g<T, W, false, true>(p, m, grid, s);
  return gemma ? launch_bwd_g<T, W, true, false>(p, m, grid, s)
               : launch_bwd_g<T, W, false, false>(p, m, grid, s);
}

cudaError_t launch_fwd_staged(const FwdArgs& a, const Mapping& m, const DeviceInfo& d,
                              long long wait_limit, cudaStream_t s) {
  const bool res = a.res != nullptr;
  rmsk::StagedParams p = params(m, a.M, a.N, res ? 2 : 1, wait_limit);
  p.x = a.x;
  p.gamma = a.gamma;
  p.out = a.y;
  p.rstd = a.rstd;
  p.eps = a.eps;
  p.in2 = a.res;
  p.h = a.h;
  int64_t grid = 0;
  cudaError_t e = grid_for(staged_kernel(a.dtype, false, m.kv, a.gemma, res), m, d, p.ntiles,
                           &grid);
  if (e != cudaSuccess) return e;
  const bool g = a.gemma != 0;
  switch (a.dtype) {
    case kBF16: return launch_fwd_t<__nv_bfloat16, __nv_bfloat16>(p, m, grid, g, res, s);
    case kF16: return launch_fwd_t<__half, __half>(p, m, grid, g, res, s);
    case kBF16W32: return launch_fwd_t<__nv_bfloat16, float>(p, m, grid, g, res, s);
    case kF16W32: return launch_fwd_t<__half, float>(p, m, grid, g, res, s);
    default: return launch_fwd_t<float, float>(p, m, grid, g, res, s);
  }
}

cudaError_t size_bwd_staged(const BwdArgs& a, const DeviceInfo& d, Mapping* m) {
  const int64_t ntiles = (a.M + m->rows_per_cta - 1) / m->rows_per_cta;
  int64_t grid = 0;
  cudaError_t e = grid_for(staged_kernel(a.dtype, true, m->kv, a.gemma, a.dh != nullptr), *m, d,
                           ntiles, &grid);
  if (e != cudaSuccess) return e;
  m->blocks = grid;
  m->partials = grid / m->cluster;  // one workspace row per unit
  return cudaSuccess;
}

cudaError_t launch_bwd_staged(const BwdArgs& a, const Mapping& m, const DeviceInfo& d,
                              long long wait_limit, cudaStream_t s) {
  (void)d;
  const bool res = a.dh != nullptr;
  rmsk::StagedParams p = params(m, a.M, a.N, res ? 3 : 2, wait_limit);
  p.x = a.x;
  p.gamma = a.gamma;
  p.rstd = const_cast<float*>(a.rstd);  // read only in the backward
  p.in2 = a.dy;
  p.in3 = a.dh;
  p.out = a.dx;
  p.ws = a.ws;
  const bool g = a.gemma != 0;
  switch (a.dtype) {
    case kBF16: return launch_bwd_t<__nv_bfloat16, __nv_bfloat16>(p, m, m.blocks, g, res, s);
    case kF16: return launch_bwd_t<__half, __half>(p, m, m.blocks, g, res, s);
    case kBF16W32: return launch_bwd_t<__nv_bfloat16, float>(p, m, m.blocks, g, res, s);
    case kF16W32: return launch_bwd_t<__half, float>(p, m, m.blocks, g, res, s);
    default: return launch_bwd_t<float, float>(p, m, m.blocks, g, res, s);
  }
}

cudaError_t take_device_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, rmsk::g_rms_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(rmsk::g_rms_device_status, &zero, sizeof(int));
    if (e != cudaSuccess) return e;
  }
  *status = v;
  return cudaSuccess;
}

}  // namespace rmsi
