// E4M3 (FP8) helpers shared by the forward kernels with a quantised output:
// the float32 -> E4M3 conversion of two values (round to nearest even,
// saturating to +-448, the instruction the hardware provides), the stored
// y of a vector widened back to float32 pairs, and the absolute maximum of
// stored vectors.
#pragma once

#include "common.cuh"

namespace rmsk {

// Two float32 values to two E4M3 codes (round to nearest even, saturating
// to the largest finite value), low element in the low byte.
__device__ __forceinline__ uint32_t f2_to_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// ss_lo += x_lo^2 and ss_hi += x_hi^2 over the element pairs of one vector:
// the float32 operations of RowMath::sumsq (one fused multiply-add per
// element on its exact float32 value), taking the 16-bit values as they are
// stored: a mixed-precision fma (16-bit factors, float32 addend and result)
// is exact in the product and rounds once, like the fma of the widened
// values, and leaves no widened copy of x to hold in registers.
template <typename T>
struct SumSqDirect {
  __device__ static __forceinline__ void add(const uint4& x, float& lo, float& hi) {
    f32x2 ss = pk2(lo, hi);
    RowMath<T, T, false>::sumsq(x, ss);
    lo = lo2(ss);
    hi = hi2(ss);
  }
};
template <>
struct SumSqDirect<__nv_bfloat16> {
  __device__ static __forceinline__ void add(const uint4& x, float& lo, float& hi) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
          "fma.rn.f32.bf16 %0, a, a, %0;\n\tfma.rn.f32.bf16 %1, b, b, %1;\n\t}"
          : "+f"(lo), "+f"(hi) : "r"(w[i]));
    }
  }
};
template <>
struct SumSqDirect<__half> {
  __device__ static __forceinline__ void add(const uint4& x, float& lo, float& hi) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
          "fma.rn.f32.f16 %0, a, a, %0;\n\tfma.rn.f32.f16 %1, b, b, %1;\n\t}"
          : "+f"(lo), "+f"(hi) : "r"(w[i]));
    }
  }
};

// The stored y of one vector widened back to float32 pairs.
template <typename T>
__device__ __forceinline__ f32x2 stored_pair(const uint4& yv, int i) {
  return Pairs<T>::get(yv, i);
}

// max |y| over one stored vector, folded into a running maximum.  For the
// 16-bit types the magnitudes are compared packed (sign bits cleared, one
// two-lane max per word); the float32 value of the result is exact.
template <typename T>
struct AbsMax;
template <>
struct AbsMax<float> {
  float m = 0.f;
  __device__ __forceinline__ void add(const uint4& v) {
    m = fmaxf(m, fmaxf(fmaxf(fabsf(__uint_as_float(v.x)), fabsf(__uint_as_float(v.y))),
                       fmaxf(fabsf(__uint_as_float(v.z)), fabsf(__uint_as_float(v.w)))));
  }
  __device__ __forceinline__ float value() const { return m; }
};
template <>
struct AbsMax<__nv_bfloat16> {
  __nv_bfloat162 m = __floats2bfloat162_rn(0.f, 0.f);
  __device__ __forceinline__ void add(const uint4& v) {
    const uint32_t w[4] = {v.x & 0x7fff7fffu, v.y & 0x7fff7fffu, v.z & 0x7fff7fffu,
                           v.w & 0x7fff7fffu};
#pragma unroll
    for (int i = 0; i < 4; ++i) m = __hmax2(m, *reinterpret_cast<const __nv_bfloat162*>(&w[i]));
  }
  __device__ __forceinline__ float value() const {
    return fmaxf(__low2float(m), __high2float(m));
  }
};
template <>
struct AbsMax<__half> {
  __half2 m = __floats2half2_rn(0.f, 0.f);
  __device__ __forceinline__ void add(const uint4& v) {
    const uint32_t w[4] = {v.x & 0x7fff7fffu, v.y & 0x7fff7fffu, v.z & 0x7fff7fffu,
                           v.w & 0x7fff7fffu};
#pragma unroll
    for (int i = 0; i < 4; ++i) m = __hmax2(m, *reinterpret_cast<const __half2*>(&w[i]));
  }
  __device__ __forceinline__ float value() const {
    return fmaxf(__low2float(m), __high2float(m));
  }
};

}  // namespace rmsk
