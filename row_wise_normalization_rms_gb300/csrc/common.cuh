// Device helpers shared by the RMSNorm kernels: element traits, 16-byte
// vector pack/unpack, streaming loads/stores and the fixed-order
// reductions every kernel uses.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

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

template <>
struct Elem<__half> {
  static constexpr int kPerVec = 8;
  __device__ static __forceinline__ float to_f(__half v) { return __half2float(v); }
  __device__ static __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
  __device__ static __forceinline__ float round(float v) { return __half2float(__float2half_rn(v)); }
  __device__ static __forceinline__ void unpack(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ static __forceinline__ uint4 pack(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// ---- packed float pairs ------------------------------------------------------
// Blackwell issues two float32 FMAs/multiplies per instruction on register
// pairs (fma.rn.f32x2 / mul.rn.f32x2): each lane is an ordinary IEEE float32
// operation with a single rounding, so results equal the scalar forms.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pk2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float lo2(f32x2 v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo;
}
__device__ __forceinline__ float hi2(f32x2 v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return hi;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 splat2(float v) { return pk2(v, v); }
// Exact negation of both halves (sign bits flipped).
__device__ __forceinline__ f32x2 neg2(f32x2 v) { return v ^ 0x8000000080000000ull; }

// Compensated (Kahan) running sums, for row reductions whose per-thread
// chains grow with N: the error stays a few units in the last place of the
// sum of magnitudes however many terms are added.  Every step is an
// explicitly rounded add, so nothing is reassociated or contracted.
struct Kahan2 {
  f32x2 s = 0ull, c = 0ull;  // sum, and the negated part lost so far
  __device__ __forceinline__ void add(f32x2 v) {
    const f32x2 y = add2(v, neg2(c));
    const f32x2 t = add2(s, y);
    c = add2(add2(t, neg2(s)), neg2(y));
    s = t;
  }
  __device__ __forceinline__ float total() const {
    const f32x2 r = add2(s, neg2(c));
    return __fadd_rn(lo2(r), hi2(r));
  }
};
struct Kahan1 {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float v) {
    const float y = __fsub_rn(v, c);
    const float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
  }
  __device__ __forceinline__ float total() const { return __fsub_rn(s, c); }
};

// Two bf16 (one 32-bit word, low half first) widened exactly to a pair.
__device__ __forceinline__ f32x2 bf2_to_f2(uint32_t w) {
  return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// A pair rounded to two bf16 (round to nearest even), low half first.
__device__ __forceinline__ uint32_t f2_to_bf2(f32x2 v) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo2(v), hi2(v));
  return *reinterpret_cast<uint32_t*>(&h);
}
// Product of two bf16 pairs rounded once to bf16.  The exact product of two
// 8-bit significands fits a float32, so this equals rounding the float32
// product of the widened values.
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Two fp16 (one 32-bit word, low half first) widened exactly to a pair.
__device__ __forceinline__ f32x2 h2_to_f2(uint32_t w) {
  const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w));
  return pk2(t.x, t.y);
}
__device__ __forceinline__ uint32_t f2_to_h2(f32x2 v) {
  __half2 h = __floats2half2_rn(lo2(v), hi2(v));
  return *reinterpret_cast<uint32_t*>(&h);
}
// Product of two fp16 pairs rounded once to fp16.  The exact product of two
// 11-bit significands (and any fp16 exponents) fits a float32 exactly, so
// this equals rounding the float32 product of the widened values.
__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The exact float32 products of two pairs of 16-bit values (one 32-bit word
// each, low half first): one mixed-precision fma per element (16-bit factors,
// float32 addend -0, which leaves every product, signed zeros included, as
// the float32 multiply of the widened values gives it; the product of two
// bf16 or two fp16 significands fits a float32 exactly).
__device__ __forceinline__ f32x2 mul_exact2(uint32_t a, uint32_t b, const __nv_bfloat16*) {
  float lo, hi;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, 0f80000000;\n\tfma.rn.f32.bf16 %1, ah, bh, 0f80000000;\n\t}"
      : "=f"(lo), "=f"(hi) : "r"(a), "r"(b));
  return pk2(lo, hi);
}
__device__ __forceinline__ f32x2 mul_exact2(uint32_t a, uint32_t b, const __half*) {
  float lo, hi;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, al, bl, 0f80000000;\n\tfma.rn.f32.f16 %1, ah, bh, 0f80000000;\n\t}"
      : "=f"(lo), "=f"(hi) : "r"(a), "r"(b));
  return pk2(lo, hi);
}

// 32-bit word i of a 16-byte vector.
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Pair conversion and the rounding weight multiply for the 16-bit types.
template <typename T>
struct Half2Ops;
template <>
struct Half2Ops<__nv_bfloat16> {
  __device__ static __forceinline__ f32x2 widen(uint32_t w) { return bf2_to_f2(w); }
  __device__ static __forceinline__ uint32_t narrow(f32x2 v) { return f2_to_bf2(v); }
  __device__ static __forceinline__ uint32_t mul(uint32_t a, uint32_t b) { return bf2_mul(a, b); }
};
template <>
struct Half2Ops<__half> {
  __device__ static __forceinline__ f32x2 widen(uint32_t w) { return h2_to_f2(w); }
  __device__ static __forceinline__ uint32_t narrow(f32x2 v) { return f2_to_h2(v); }
  __device__ static __forceinline__ uint32_t mul(uint32_t a, uint32_t b) { return h2_mul(a, b); }
};

// A 16-byte vector as float pairs: 4 pairs for bf16 and fp16, 2 for float32.
template <typename T>
struct Pairs;
template <>
struct Pairs<__nv_bfloat16> {
  static constexpr int n = 4;
  __device__ static __forceinline__ f32x2 get(const uint4& v, int i) {
    return bf2_to_f2(i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w);
  }
};
template <>
struct Pairs<__half> {
  static constexpr int n = 4;
  __device__ static __forceinline__ f32x2 get(const uint4& v, int i) {
    return h2_to_f2(i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w);
  }
};
template <>
struct Pairs<float> {
  static constexpr int n = 2;
  __device__ static __forceinline__ f32x2 get(const uint4& v, int i) {
    return i == 0 ? pk2(__uint_as_float(v.x), __uint_as_float(v.y))
                  : pk2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
};

// ---- the weight beside one activation vector ----------------------------------
// The weight values of the columns of one 16-byte activation vector: one
// vector when the weight has the activations' type, two float32 vectors when
// a 16-bit activation comes with a float32 weight.
template <typename T>
struct GammaSame {
  uint4 v;
  __device__ static __forceinline__ GammaSame load(const void* gamma, int vec) {
    return GammaSame{__ldg(reinterpret_cast<const uint4*>(gamma) + vec)};
  }
  __device__ static __forceinline__ GammaSame zero() { return GammaSame{make_uint4(0u, 0u, 0u, 0u)}; }
  __device__ __forceinline__ f32x2 pair(int i) const { return Pairs<T>::get(v, i); }
  // 32-bit word i: two 16-bit weights, for the packed 16-bit multiply.
  __device__ __forceinline__ uint32_t word(int i) const {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
  }
};

// Eight float32 weights beside one vector of eight 16-bit activations.
struct GammaW32 {
  uint4 a, b;  // weights of elements 0..3 and 4..7
  __device__ static __forceinline__ GammaW32 load(const void* gamma, int vec) {
    const uint4* g = reinterpret_cast<const uint4*>(gamma) + 2 * vec;
    return GammaW32{__ldg(g), __ldg(g + 1)};
  }
  __device__ static __forceinline__ GammaW32 zero() {
    return GammaW32{make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
  }
  __device__ __forceinline__ f32x2 pair(int i) const {
    const uint4& q = i < 2 ? a : b;
    return (i & 1) ? pk2(__uint_as_float(q.z), __uint_as_float(q.w))
                   : pk2(__uint_as_float(q.x), __uint_as_float(q.y));
  }
  __device__ __forceinline__ uint32_t word(int) const { return 0u; }  // not used with W32
};

template <typename T, typename W>
struct GammaSel {
  using type = GammaSame<T>;
};
template <>
struct GammaSel<__nv_bfloat16, float> {
  using type = GammaW32;
};
template <>
struct GammaSel<__half, float> {
  using type = GammaW32;
};
template <typename T, typename W>
using GammaVec = typename GammaSel<T, W>::type;

// ---- per-vector arithmetic ---------------------------------------------------
#ifndef RMS_MIXED_U
#define RMS_MIXED_U 1
#endif
// Shared by every vector kernel, so all mappings compute identical bits.
// T: activation type; W: weight type (T, or float with 16-bit T).
template <typename T, typename W, bool GEMMA>
struct RowMath {
  using P = Pairs<T>;
  using G = GammaVec<T, W>;
  static constexpr int kPairs = P::n;

  // Effective weight pair: gamma, or 1 + gamma (Gemma).
  __device__ static __forceinline__ f32x2 weight(const G& g, int i) {
    const f32x2 w = g.pair(i);
    return GEMMA ? add2(w, splat2(1.0f)) : w;
  }

  // u = dy * weight for element pair i.  With 16-bit dy and weight (not
  // Gemma) the exact product is taken from the stored values by
  // mixed-precision fma, without widening either; otherwise the float32
  // multiply of the widened values (the same bits).
  static constexpr bool kMixedU = RMS_MIXED_U && sizeof(T) == 2 && sizeof(W) == 2 && !GEMMA;
  __device__ static __forceinline__ f32x2 u_pair(const uint4& dy, const G& g, int i) {
    if constexpr (kMixedU) {
      return mul_exact2(word_of(dy, i), g.word(i), (const T*)nullptr);
    } else {
      return mul2(P::get(dy, i), weight(g, i));
    }
  }

  // ss += x^2 over the vector.
  __device__ static __forceinline__ void sumsq(const uint4& x, f32x2& ss) {
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      const f32x2 f = P::get(x, i);
      ss = fma2(f, f, ss);
    }
  }

  // y for one vector.  Non-Gemma: (x*r) rounded to the weight type, then
  // times gamma, rounded to the output type (with a float32 weight the first
  // rounding is exact).  Gemma: x*r*(1+gamma) rounded once.
  __device__ static __forceinline__ uint4 forward(const uint4& x, const G& g, float r) {
    const f32x2 rr = splat2(r);
    uint32_t o[4];
    if constexpr (sizeof(T) == 2) {
      using H = Half2Ops<T>;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const f32x2 xr = mul2(P::get(x, i), rr);
        if constexpr (GEMMA || sizeof(W) == 4) {
          o[i] = H::narrow(mul2(xr, weight(g, i)));
        } else {
          o[i] = H::mul(H::narrow(xr), g.word(i));
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const f32x2 y = mul2(mul2(P::get(x, i), rr), weight(g, i));
        o[2 * i] = __float_as_uint(lo2(y));
        o[2 * i + 1] = __float_as_uint(hi2(y));
      }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  }

  // Backward first pass over one vector, with xn = x*r and u = dy*w:
  // sux += u*xn (the row's r*sum(u*x)) and acc += dy*xn (dgamma terms).
  __device__ static __forceinline__ void backward_sums(const uint4& x, const uint4& dy, const G& g,
                                                       float r, f32x2& sux, f32x2* acc) {
    const f32x2 rr = splat2(r);
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      const f32x2 xn = mul2(P::get(x, i), rr);
      const f32x2 d = P::get(dy, i);
      sux = fma2(kMixedU ? u_pair(dy, g, i) : mul2(d, weight(g, i)), xn, sux);
      acc[i] = fma2(d, xn, acc[i]);
    }
  }

  // The two halves of backward_sums, for mappings that take them in
  // separate passes: sux += u*xn, and acc += dy*xn.
  __device__ static __forceinline__ void backward_dot(const uint4& x, const uint4& dy, const G& g,
                                                      float r, f32x2& sux) {
    const f32x2 rr = splat2(r);
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      const f32x2 xn = mul2(P::get(x, i), rr);
      sux = fma2(u_pair(dy, g, i), xn, sux);
    }
  }
  __device__ static __forceinline__ void backward_acc(const uint4& x, const uint4& dy, float r,
                                                      f32x2* acc) {
    const f32x2 rr = splat2(r);
#pragma unroll
    for (int i = 0; i < kPairs; ++i) acc[i] = fma2(P::get(dy, i), mul2(P::get(x, i), rr), acc[i]);
  }

  // dx for one vector: r*u - x*r^3*c = r*(u - xn*k) with k = r*c.
  __device__ static __forceinline__ uint4 backward_dx(const uint4& x, const uint4& dy, const G& g,
                                                      float r, float k) {
    const f32x2 rr = splat2(r);
    const f32x2 nk = splat2(-k);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      const f32x2 xn = mul2(P::get(x, i), rr);
      const f32x2 u = u_pair(dy, g, i);
      const f32x2 dx = mul2(fma2(xn, nk, u), rr);
      if constexpr (sizeof(T) == 2) {
        o[i] = Half2Ops<T>::narrow(dx);
      } else {
        o[2 * i] = __float_as_uint(lo2(dx));
        o[2 * i + 1] = __float_as_uint(hi2(dx));
      }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  }

  // The same dx with the gradient dh reaching the same input through a
  // residual path added in float32 before the one rounding.
  __device__ static __forceinline__ uint4 backward_dx_add(const uint4& x, const uint4& dy,
                                                          const G& g, float r, float k,
                                                          const uint4& dh) {
    const f32x2 rr = splat2(r);
    const f32x2 nk = splat2(-k);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      const f32x2 xn = mul2(P::get(x, i), rr);
      const f32x2 u = u_pair(dy, g, i);
      const f32x2 dx = add2(mul2(fma2(xn, nk, u), rr), P::get(dh, i));
      if constexpr (sizeof(T) == 2) {
        o[i] = Half2Ops<T>::narrow(dx);
      } else {
        o[2 * i] = __float_as_uint(lo2(dx));
        o[2 * i + 1] = __float_as_uint(hi2(dx));
      }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  }

  // h = x + residual for one vector: float32 sum, one rounding to the
  // activation type (the residual stream keeps that type).
  __device__ static __forceinline__ uint4 add_round(const uint4& a, const uint4& b) {
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      const f32x2 h = add2(P::get(a, i), P::get(b, i));
      if constexpr (sizeof(T) == 2) {
        o[i] = Half2Ops<T>::narrow(h);
      } else {
        o[2 * i] = __float_as_uint(lo2(h));
        o[2 * i + 1] = __float_as_uint(hi2(h));
      }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  }
};

// ---- memory ----------------------------------------------------------------
// Rows are touched once per kernel: load and store them evict-first so they
// do not push gamma and the partial sums out of L2.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) { __stcs(p, v); }
__device__ __forceinline__ uint4 ld_keep(const uint4* p) { return __ldg(p); }

// ---- programmatic dependent launch ------------------------------------------
// Every kernel is launched with programmatic stream serialisation allowed,
// so it may be scheduled while its predecessor in the stream is finishing,
// and waits for the predecessor's completion and memory (pdl_wait) before it
// reads or writes any global memory.  Only the non-persistent forward
// kernels let their dependents be scheduled early (pdl_trigger, once every
// CTA has started); the persistent kernels trigger implicitly at exit: an
// early trigger there let dependents take SM slots mid-run and cost up to
// 50 % at some shapes.  Both are no-ops without such a dependency.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// Sum over an aligned group of G lanes of one warp (G a power of two up to
// 32), butterfly order: every lane of the group gets the same bits.
__device__ __forceinline__ float lane_group_sum(float v, int G) {
  for (int o = G >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Host side: launch `kernel` with programmatic stream serialisation allowed.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace rmsk
