// Element-wise access to row vectors as fp32 lanes (fp32 or bf16 rows).
#pragma once

#include "common.cuh"

namespace moe {

// 32-bit words of a vector.
template <typename V> struct Words;
template <> struct Words<u32x8> {
  static constexpr int N = 8;
  __device__ __forceinline__ static uint32_t get(const u32x8& v, int i) { return v.w[i]; }
  __device__ __forceinline__ static void set(u32x8& v, int i, uint32_t w) { v.w[i] = w; }
};
template <> struct Words<uint4> {
  static constexpr int N = 4;
  __device__ __forceinline__ static uint32_t get(const uint4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
  }
  __device__ __forceinline__ static void set(uint4& v, int i, uint32_t w) {
    if (i == 0) v.x = w; else if (i == 1) v.y = w; else if (i == 2) v.z = w; else v.w = w;
  }
};
template <> struct Words<uint2> {
  static constexpr int N = 2;
  __device__ __forceinline__ static uint32_t get(const uint2& v, int i) { return i == 0 ? v.x : v.y; }
  __device__ __forceinline__ static void set(uint2& v, int i, uint32_t w) { if (i == 0) v.x = w; else v.y = w; }
};
template <> struct Words<uint32_t> {
  static constexpr int N = 1;
  __device__ __forceinline__ static uint32_t get(const uint32_t& v, int) { return v; }
  __device__ __forceinline__ static void set(uint32_t& v, int, uint32_t w) { v = w; }
};

// A vector of VB bytes holding elements of type ET, read and written as fp32.
template <int VB, typename ET> struct Lanes {
  using V = typename Vec<VB>::T;
  static constexpr int kElems = VB / Elem<ET>::kBytes;
  __device__ __forceinline__ static float get(const V& v, int q) {
    if constexpr (Elem<ET>::kBytes == 4) {
      return __uint_as_float(Words<V>::get(v, q));
    } else {
      return Elem<ET>::get(Words<V>::get(v, q >> 1), q & 1);
    }
  }
  __device__ __forceinline__ static V pack(const float* a) {
    V v;
    if constexpr (Elem<ET>::kBytes == 4) {
#pragma unroll
      for (int q = 0; q < Words<V>::N; ++q) Words<V>::set(v, q, __float_as_uint(a[q]));
    } else {
#pragma unroll
      for (int q = 0; q < Words<V>::N; ++q) Words<V>::set(v, q, pack_bf16x2(a[2 * q], a[2 * q + 1]));
    }
    return v;
  }
};

// A single bf16 element (rows whose byte length is not a multiple of 4).
template <> struct Lanes<2, __nv_bfloat16> {
  using V = uint16_t;
  static constexpr int kElems = 1;
  __device__ __forceinline__ static float get(const V& v, int) { return __uint_as_float((uint32_t)v << 16); }
  __device__ __forceinline__ static V pack(const float* a) {
    __nv_bfloat16 b = __float2bfloat16_rn(a[0]);
    return *reinterpret_cast<uint16_t*>(&b);
  }
};

}  // namespace moe

namespace moe {

// Two fp32 values in one 64-bit register, operated on by Blackwell's packed
// f32x2 instructions (each half rounded to nearest, like __fadd_rn /
// __fmul_rn; subnormals kept).
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  uint32_t a, b;
  asm("mov.b64 {%0,%1}, %2;" : "=r"(a), "=r"(b) : "l"(v));
  lo = __uint_as_float(a);
  hi = __uint_as_float(b);
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// Word q of a vector as an fp32 pair: two bf16 elements (low first) or, for
// fp32 rows, elements 2q and 2q+1.
template <typename ET, typename V>
__device__ __forceinline__ uint64_t f2_elems(const V& v, int q) {
  if constexpr (Elem<ET>::kBytes == 2) {
    const uint32_t w = Words<V>::get(v, q);
    return f2_pack(w << 16, w & 0xffff0000u);
  } else {
    return f2_pack(Words<V>::get(v, 2 * q), Words<V>::get(v, 2 * q + 1));
  }
}

}  // namespace moe
