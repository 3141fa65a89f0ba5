// Device helpers shared by the RMSNorm kernels: element traits, 16-byte
// vector pack/unpack, streaming loads/stores and the fixed-order
// reductions every kernel uses.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsk {

// ---- element traits --------------------------------------------------------
// Every value is widened to float32 on load and rounded once (round to
// nearest even) on store.
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kPerVec = 4;  // elements per 16-byte vector
  __device__ static __forceinline__ float to_f(float v) { return v; }
  __device__ static __forceinline__ float from_f(float v) { return v; }
  // Rounding to the I/O type (identity for float32).
  __device__ static __forceinline__ float round(float v) { return v; }
  __device__ static __forceinline__ void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static __forceinline__ uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kPerVec = 8;
  __device__ static __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ static __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
  __device__ static __forceinline__ float round(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
  }
  // bf16 -> f32 widening is exact: the 16 bits become the high half.
  __device__ static __forceinline__ void unpack(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static __forceinline__ uint4 pack(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// ---- memory ----------------------------------------------------------------
// Rows are touched once per kernel: load and store them evict-first so they
// do not push gamma and the partial sums out of L2.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) { __stcs(p, v); }
__device__ __forceinline__ uint4 ld_keep(const uint4* p) { return __ldg(p); }

// ---- reductions ------------------------------------------------------------
// Butterfly sum over a warp.  a+b == b+a exactly, so every lane ends with the
// same bits and the order depends on nothing but the lane layout.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum of `v` over a group of G threads (G a multiple of 32) that occupy
// warps [first_warp, first_warp + G/32) of the CTA.  `red` holds one float
// per warp of the CTA.  Every thread of the CTA must call this (it contains
// a __syncthreads when G > 32).  The cross-warp sum runs in warp order, so
// the result is deterministic.  Callers that reuse `red` for the next row
// must alternate between two buffers.
__device__ __forceinline__ float group_sum(float v, int G, int first_warp, float* red) {
  v = warp_sum(v);
  if (G == 32) return v;
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
  const int nw = G >> 5;
  for (int w = 0; w < nw; ++w) s += red[first_warp + w];
  return s;
}

}  // namespace rmsk
